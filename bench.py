"""Benchmark of the tiled fp32 maps on GB300.

One step is one pass of the whole hot path over one batch: the fp32
[8192, 8192] matrix X ~ N(0,1) (seed 1) of the aligned 2-D scale workload
("@aligned", "A minimal kernel": TM = 32, TN = 128), fed through every kernel:

  affine      out = X*2 + 1 over all 67,108,864 elements (1-D, widest vectors)
  scale2d     Y = 1.5*X, 32 x 128 tiles, aligned promise
  copy2d      B = X, 64 x 64 tiles, aligned promise
  rowsum      r = sum over each row (a block per row, 1024-column tiles)
  colsum      c = sum over each column (32 x 128 strips, AUTO variant: one
              pass of 8-CTA thread-block clusters, a strip's partials added
              over distributed shared memory)
  rowmax      m = ragged row max (a block per row), 64-column tiles, -inf fill

Metric: achieved HBM GB/s (GB = 1e9 bytes, the pages' convention) over the
algorithmic bytes (each input byte read once, each output byte written once),
and its fraction of the measured HBM peak.  Inputs are larger than L2 (256 MiB
vs 126 MB), so no flush runs between steps.  The JSON line also carries
`configs`: every kernel on the workload its target is stated on (the 1M
affine map, the aligned and ragged 2-D maps, the 64 MB row and column sums,
the ragged row max), a lone launch after an L2 flush and back-to-back
overlapped launches, each output checked against the oracle first.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--sweep]
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s and % of GB300 HBM roofline per kernel (1 GPU)"
WORKLOAD = "scale_8192"
M = N = 8192
ALPHA = 1.5
FALLBACK_HBM_GBS = 6800.0
STEP_LAUNCHES = 6  # affine, scale2d, copy2d, rowsum, colsum (AUTO: one pass of 8-CTA clusters here), rowmax
ROWSUM_TILE = (1, 1024)   # rows per block x columns per tile
COLSUM_TILE = (32, 128)   # row tile x column strip
ROWMAX_BR = 1             # rows per block (column tile BC = 64)


def gbps(nbytes: int, seconds: float) -> float:
    """Bandwidth in GB/s with GB = 1e9 bytes (the pages' convention: their
    "64 MB" read in 111.6 us is quoted as 601 GB/s, i.e. 2^26 bytes / 1e9)."""
    return nbytes / seconds / 1e9


def kernel_bytes(M: int, N: int) -> dict:
    """Algorithmic bytes of each kernel of one step over an [M, N] fp32 batch."""
    e = M * N
    return {
        "affine": 8 * e,
        "scale2d": 8 * e,
        "copy2d": 8 * e,
        "rowsum": 4 * e + 4 * M,
        "colsum": 4 * e + 4 * N,
        "rowmax_masked": 4 * e + 4 * M,
    }


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs: torch copy of 1 Gi bf16, read+write)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, an earlier GB300 measurement)"


def aggregate(elapsed_s: float, nbytes: int, world: int):
    """Max of the ranks' elapsed times and sum of their bytes (torch.distributed
    when world > 1; the process group must be initialised)."""
    if world <= 1:
        return elapsed_s, nbytes
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed_s], dtype=torch.float64)
    b = torch.tensor([float(nbytes)], dtype=torch.float64)
    if dist.get_backend() == "nccl":
        t, b = t.cuda(), b.cuda()
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), int(b.item())


# --------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 200 ms) while the timed region runs."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        inside = [r for (t, r) in self.rows if t0 <= t <= t1 + 0.25]
        rows = inside or [r for (_, r) in self.rows]
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows if len(r) >= 9 for k in range(4) if r[5 + k] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "samples_in_timed_region": len(inside)}


# --------------------------------------------------------------------- traffic
def traffic_source():
    """Where and when the committed DRAM-traffic figures were captured."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            return json.load(f).get("_captured")
    except Exception:
        return None


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, when it was taken
    on the current source of that kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    ent = rec.get(kernel)
    if not ent:
        return None
    src = os.path.join(ROOT, "masking_tm_affine_gb300", "csrc", ent["source"])
    try:
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    if digest != ent.get("source_sha256_16"):
        return None
    return ent.get("dram_bytes_per_launch_full")


# --------------------------------------------------------------------- GPU arm
def make_step(tm, bufs, ws_bytes, stream, overlap=True, first_overlap=True):
    """The hot path over one batch, as (name, launch) pairs on `stream`.

    overlap: every call is an overlapped launch (TM_PDL), which may start while
    the previous call's kernel drains.  The contract holds: all six calls read
    only X, which no call writes, and every store still waits for the previous
    kernel.  first_overlap=False launches the first call plainly, for a step
    whose X has just been copied in by another stream."""
    X, A1, Y, B, r, c, m, W = (bufs[k] for k in ("X", "A1", "Y", "B", "r", "c", "m", "W"))
    s = stream.cuda_stream
    P = tm.TM_PDL if overlap else 0
    P0 = P if first_overlap else 0
    return [
        ("affine", lambda: tm.tm_affine(X, A1, M * N, tm.TM_VAR_AUTO | P0, s)),
        ("scale2d", lambda: tm.tm_scale2d(X, N, Y, N, M, N, ALPHA, 32, 128, tm.TM_ALIGNED | P, s)),
        ("copy2d", lambda: tm.tm_copy2d(X, N, B, N, M, N, 64, 64, tm.TM_ALIGNED | P, s)),
        ("rowsum", lambda: tm.tm_rowsum(X, N, M, N, r, *ROWSUM_TILE, tm.TM_ALIGNED | P, s)),
        ("colsum", lambda: tm.tm_colsum(X, N, M, N, c, W, ws_bytes, *COLSUM_TILE, tm.TM_VAR_AUTO,
                                        tm.TM_ALIGNED | P, s)),
        ("rowmax_masked", lambda: tm.tm_rowmax_masked(X, N, M, N, m, ROWMAX_BR, 64, tm.TM_FILL_NEG_INF,
                                                      tm.TM_ALIGNED | P, s)),
    ]


def make_buffers(tm, x, dev):
    """Device buffers of one step over the batch x ([M, N] fp32 on the host)."""
    import torch
    bufs = {
        "X": torch.from_numpy(x.reshape(-1)).to(dev),
        "A1": torch.empty(M * N, dtype=torch.float32, device=dev),
        "Y": torch.empty(M * N, dtype=torch.float32, device=dev),
        "B": torch.empty(M * N, dtype=torch.float32, device=dev),
        "r": torch.empty(M, dtype=torch.float32, device=dev),
        "c": torch.empty(N, dtype=torch.float32, device=dev),
        "m": torch.empty(M, dtype=torch.float32, device=dev),
    }
    ws_bytes = tm.tm_colsum_workspace_bytes(M, N, *COLSUM_TILE)
    bufs["W"] = torch.empty(max(ws_bytes // 4, 4), dtype=torch.float32, device=dev)
    return bufs, ws_bytes


def verify_step(bufs, x, oracle, rows=None):
    """Parity of one step at full size against the oracle: the given rows of
    every output (default 64 rows spread over the batch; `rows="all"` for
    every row), and every column sum."""
    import numpy as np
    if rows is None:
        rows = np.linspace(0, M - 1, 64).astype(np.int64)
    elif isinstance(rows, str):
        rows = np.arange(M, dtype=np.int64)
    xs = x[rows]
    A1 = bufs["A1"].view(M, N)[rows].cpu().numpy()
    Y = bufs["Y"].view(M, N)[rows].cpu().numpy()
    B = bufs["B"].view(M, N)[rows].cpu().numpy()
    assert np.array_equal(A1.view(np.uint32), oracle.affine(xs).reshape(xs.shape).view(np.uint32)), "affine"
    want = np.zeros_like(xs)
    oracle.scale2d(xs, N, want, N, len(rows), N, ALPHA)
    assert np.array_equal(Y.view(np.uint32), want.view(np.uint32)), "scale2d"
    want_b = np.zeros(xs.size, dtype=np.uint32)
    oracle.copy2d(xs, N, want_b, N, len(rows), N)
    assert np.array_equal(B.view(np.uint32).reshape(-1), want_b), "copy2d"
    r = bufs["r"].cpu().numpy()[rows]
    rw = oracle.rowsum(xs, N, len(rows), N)
    assert np.all(np.abs(r - rw) <= 1e-5 * oracle.rowsum(np.abs(xs), N, len(rows), N)), "rowsum"
    c = bufs["c"].cpu().numpy()
    cw = oracle.colsum(x, N, M, N)
    assert np.all(np.abs(c - cw) <= 1e-5 * oracle.colsum(np.abs(x), N, M, N)), "colsum"
    mm = bufs["m"].cpu().numpy()[rows]
    assert np.array_equal(mm, oracle.rowmax_masked(xs, N, len(rows), N, 64)), "rowmax"


def cpu_baseline(x, budget_s: float = 12.0) -> dict:
    """The oracle as it stands, one thread pinned to one core, over a bounded
    sample: rows [0, 1024) of the batch, whole passes until ~budget_s."""
    import numpy as np
    import oracle
    oracle.build()
    R = 1024
    xs = np.ascontiguousarray(x[:R])
    by = sum(kernel_bytes(R, N).values())
    prev = os.sched_getaffinity(0) if hasattr(os, "sched_getaffinity") else None
    if prev:
        os.sched_setaffinity(0, {min(prev)})
    try:
        Yw = np.empty_like(xs)
        Bw = np.empty(xs.size, dtype=np.uint32)

        def one_pass():
            oracle.affine(xs)
            oracle.scale2d(xs, N, Yw, N, R, N, ALPHA)
            oracle.copy2d(xs, N, Bw, N, R, N)
            oracle.rowsum(xs, N, R, N)
            oracle.colsum(xs, N, R, N)
            oracle.rowmax_masked(xs, N, R, N, 64)

        one_pass()  # warm-up
        t0 = time.perf_counter()
        passes = 0
        while True:
            one_pass()
            passes += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                break
    finally:
        if prev:
            os.sched_setaffinity(0, prev)
    return {"value": round(gbps(by * passes, el), 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": "oracle step (all six maps) over rows [0,%d) of the [8192,8192] batch, %d passes in "
                      "%.1f s, single thread pinned to one core of %d" % (R, passes, el, os.cpu_count())}


def run_gpu(args):
    import numpy as np
    import torch

    from masking_tm_affine_gb300 import synth, tm

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    tm.load()

    x = synth.workload_input(WORKLOAD)
    bufs, ws_bytes = make_buffers(tm, x, dev)
    stream = torch.cuda.Stream(device=dev)
    step = make_step(tm, bufs, ws_bytes, stream)
    plain = make_step(tm, bufs, ws_bytes, stream, overlap=False)
    names = [n for n, _ in step]
    kb = kernel_bytes(M, N)
    step_bytes = sum(kb.values())

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 1)):
            for _, fn in step:
                fn()
        tm.tm_check(stream.cuda_stream)
    if rank == 0 and not args.no_verify:
        import oracle
        oracle.build()
        verify_step(bufs, x, oracle)

    # timed region: K steps of overlapped launches, one event pair around them
    # (an event between two kernels would end the overlap), barrier and
    # synchronize on both sides.  The region runs again until at least
    # --min-timed-s have passed (and at least 3 times), so the clock sampler
    # sees the GPU under this load; `value` comes from the median region.
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.6)

    def region():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for k in range(args.steps):
                for _, fn in step:
                    fn()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        return e0.elapsed_time(e1) * 1e-3

    wall0 = time.time()
    regions = [region()]
    n_regions = max(3, int(args.min_timed_s / max(regions[0], 1e-6)) + 1)
    if world > 1:  # every rank runs the same number of regions
        nr = torch.tensor([n_regions], dtype=torch.int64, device=dev)
        torch.distributed.all_reduce(nr, op=torch.distributed.ReduceOp.MAX)
        n_regions = int(nr.item())
    while len(regions) < n_regions:
        regions.append(region())
    wall1 = time.time()
    tm.tm_check(stream.cuda_stream)
    elapsed = statistics.median(regions)

    # per-kernel pass: the same K steps launched plainly, an event pair around
    # every launch, for each kernel's own duration (the roofline's denominator)
    kp = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(plain) + 1)] for _ in range(kp)]
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for k in range(kp):
            evs[k][0].record(stream)
            for i, (_, fn) in enumerate(plain):
                fn()
                evs[k][i + 1].record(stream)
    torch.cuda.synchronize(dev)
    sampler.stop()
    tm.tm_check(stream.cuda_stream)
    plain_s = evs[0][0].elapsed_time(evs[-1][-1]) * 1e-3 / kp
    per_kernel_s = {n: sum(evs[k][i].elapsed_time(evs[k][i + 1]) for k in range(kp)) * 1e-3 / kp
                    for i, n in enumerate(names)}
    t_max, total_bytes = aggregate(elapsed, step_bytes * args.steps, world)

    # end to end through the C ABI: pinned host X in, every output back to pinned host memory
    e2e = None
    if rank == 0 and args.e2e_steps > 0:
        e2e = run_e2e(tm, bufs, x, make_step(tm, bufs, ws_bytes, stream, first_overlap=False), stream, dev,
                      min(args.steps, args.e2e_steps), step_bytes, ws_bytes, args.e2e_mode)

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return None

    peak, peak_src = measured_peak()
    configs = None
    if rank == 0 and not args.no_configs:
        configs = run_configs(tm, dev, peak, reps=args.reps, verify=not args.no_verify, x_step=x)
    kernels = {}
    for n in names:
        t = per_kernel_s[n]
        a = gbps(kb[n], t)
        kernels[n] = {"bytes": kb[n], "us": round(t * 1e6, 2), "GBps": round(a, 1), "frac": round(a / peak, 4)}
    dom = max(names, key=lambda n: per_kernel_s[n])
    dom_ach = gbps(kb[dom], per_kernel_s[dom])
    line = {
        "metric": METRIC,
        "value": round(gbps(total_bytes, t_max), 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_max / args.steps * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic: numpy PCG64, X ~ N(0,1) seed 1, rounded once to fp32",
        "config": {
            "workload": "scale_8192: fp32 [8192,8192] X~N(0,1) seed 1; one step = affine(1-D, all elements) + "
                        "scale2d(alpha 1.5, 32x128, aligned) + copy2d(64x64, aligned) + rowsum(%dx%d) + "
                        "colsum(%dx%d, AUTO) + rowmax_masked(%dx64, -inf fill)"
                        % (ROWSUM_TILE + COLSUM_TILE + (ROWMAX_BR,)),
            "M": M, "N": N, "step_bytes": step_bytes,
            "l2": "inputs larger than L2 (X 256 MiB, each output 256 MiB vs 126 MB L2); no flush between steps",
            "launch": "overlapped: every call passes TM_PDL (programmatic dependent launch), so a kernel's "
                      "first loads of X overlap the previous kernel's tail; stores still wait for it",
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(dom_ach, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(dom_ach / peak, 4),
                     "traffic": recorded_traffic(dom), "traffic_source": traffic_source(),
                     "peak_source": peak_src + ", of measured" if peak_src.startswith("measured") else peak_src},
        "timed_regions": {"count": len(regions), "median_ms": round(elapsed * 1e3, 4),
                          "min_ms": round(min(regions) * 1e3, 4), "max_ms": round(max(regions) * 1e3, 4),
                          "how": "the K-step region (barrier, synchronize, one event pair, K steps, synchronize) "
                                 "run back to back until >= %.1f s had passed; value and ms_per_step are the "
                                 "median region's, gpu_launches counts one region" % args.min_timed_s},
        "kernels": kernels,
        "configs": configs,
        "kernel_pass": {"ms_per_step": round(plain_s * 1e3, 4), "GBps": round(gbps(step_bytes, plain_s), 1),
                        "steps": kp, "how": "the same steps launched plainly, an event pair around every launch: "
                                            "the source of `kernels` and of the roofline's duration"},
        "gpu_launches": STEP_LAUNCHES * args.steps,
        "clocks": sampler.summary(wall0, wall1),
        "e2e": e2e,
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(x)
    if world > 1:
        torch.distributed.destroy_process_group()
    return line


def run_e2e(tm, bufs, x, step, stream, dev, steps, step_bytes, ws_bytes, mode="pipelined"):
    """The step end to end through the C ABI: every step copies its input X from
    pinned host memory and every output back to pinned host memory.

    mode "serial": copy in, six calls, copy out, one stream.
    mode "pipelined": two device buffer sets; step k's copy-in, kernels and
    copy-out run on three streams ordered by events, so step k+1's upload and
    step k-1's download overlap step k's kernels (copies of opposite directions
    also overlap on the link).  Each step still moves all of its own data."""
    import torch
    outs = ["A1", "Y", "B", "r", "c", "m"]
    hx = torch.from_numpy(x.reshape(-1)).pin_memory()
    h2d = hx.numel() * 4
    d2h = sum(bufs[k].numel() * 4 for k in outs)
    if mode == "serial":
        host = {k: torch.empty(bufs[k].numel(), dtype=torch.float32).pin_memory() for k in outs}

        def one(k):
            bufs["X"].copy_(hx, non_blocking=True)
            for _, fn in step:
                fn()
            for o in outs:
                host[o].copy_(bufs[o], non_blocking=True)
        with torch.cuda.stream(stream):
            for k in range(2):
                one(k)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for k in range(steps):
                one(k)
            e1.record(stream)
        torch.cuda.synchronize(dev)
        t = e0.elapsed_time(e1) * 1e-3
    else:
        link = measure_link(hx, bufs["X"], bufs["A1"], dev)
        link.update(measure_step_copies(hx, bufs, outs, dev))
        sets = [bufs, make_buffers(tm, x, dev)[0]]
        steps_of = [step, make_step(tm, sets[1], ws_bytes, stream, first_overlap=False)]
        hosts = [{k: torch.empty(bufs[k].numel(), dtype=torch.float32).pin_memory() for k in outs} for _ in range(2)]
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev = lambda: torch.cuda.Event()
        loaded = [ev(), ev()]
        computed = [ev(), ev()]
        drained = [ev(), ev()]
        first = [True, True]

        def one(k):
            b = k % 2
            with torch.cuda.stream(s_in):
                if not first[b]:
                    s_in.wait_event(computed[b])       # the kernels of step k-2 are done with X[b]
                sets[b]["X"].copy_(hx, non_blocking=True)
                loaded[b].record(s_in)
            with torch.cuda.stream(stream):
                stream.wait_event(loaded[b])
                if not first[b]:
                    stream.wait_event(drained[b])      # the outputs of step k-2 have left the device
                for _, fn in steps_of[b]:
                    fn()
                computed[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(computed[b])
                for o in outs:
                    hosts[b][o].copy_(sets[b][o], non_blocking=True)
                drained[b].record(s_out)
            first[b] = False
        for k in range(2):
            one(k)
        torch.cuda.synchronize(dev)
        # One continuous pipeline of (1 + nseg) segments of `seg` steps, a
        # timing event on the download stream each time a segment's last
        # outputs have left the device.  The first segment fills the pipeline
        # and is not counted; the step time is the median segment's (the host
        # side of the link may be shared with other work on the machine: a
        # stretch of ~0.1 - 0.3 s now and then runs ~60 % slower).
        seg, nseg = max(1, steps // 3), 12
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(nseg + 1)]
        for k in range(seg * (nseg + 1)):
            one(k)
            if (k + 1) % seg == 0:
                with torch.cuda.stream(s_out):
                    marks[(k + 1) // seg - 1].record(s_out)
        torch.cuda.synchronize(dev)
        segments = [marks[i].elapsed_time(marks[i + 1]) * 1e-3 / seg for i in range(nseg)]
        t = statistics.median(segments) * steps
    out = {"value": round(gbps(step_bytes * steps, t), 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": round(t / steps * 1e3, 3), "mode": mode,
           "path": "pinned host X -> device, the six C-ABI calls, every output -> pinned host"
                   + (", one stream" if mode == "serial" else
                      "; copy-in, kernels and copy-out of consecutive steps overlap on three streams")}
    if mode != "serial":
        out["segments_ms_per_step"] = [round(r * 1e3, 3) for r in segments]
        out["timing"] = ("one continuous pipeline: %d segments of %d steps after one that fills it; the median "
                         "segment's time per step" % (nseg, seg))
        floor = link_floor_s(h2d, d2h, link)
        out["link"] = {**link, "floor_ms_per_step": round(floor * 1e3, 3),
                       "frac_of_floor": round(floor / (t / steps), 4),
                       "frac_of_copies_alone": round(link["copies_alone_ms_per_step"] * 1e-3 / (t / steps), 4)}
    return out


def measure_step_copies(hx, bufs, outs, dev, reps=5):
    """One step's own copies and nothing else: X in on one stream while every
    output goes out on another (median of `reps`, after one untimed).  The
    pipelined e2e step cannot beat this: its kernels run beside the copies."""
    import torch
    host = {k: torch.empty(bufs[k].numel(), dtype=torch.float32).pin_memory() for k in outs}
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def once():
        ev = torch.cuda.Event()
        ev.record(s1)
        s2.wait_event(ev)
        with torch.cuda.stream(s1):
            bufs["X"].copy_(hx, non_blocking=True)
        with torch.cuda.stream(s2):
            for k in outs:
                host[k].copy_(bufs[k], non_blocking=True)
        s1.wait_stream(s2)

    once()
    torch.cuda.synchronize(dev)
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s1)
        once()
        e1.record(s1)
        torch.cuda.synchronize(dev)
        ts.append(e0.elapsed_time(e1) * 1e-3)
    del host
    return {"copies_alone_ms_per_step": round(statistics.median(ts) * 1e3, 3),
            "copies_alone_how": "X in and every output out, concurrently on two streams, no kernels"}


def link_floor_s(h2d_bytes, d2h_bytes, link):
    """Seconds a step needs at least to move its bytes over the host link: each
    direction at its own measured rate, and both together at the two-way
    rate (GB/s figures of `measure_link`).  A lower bound: the link may not
    reach it for an uneven mix (the step's own copies, timed alone, say what
    it does reach)."""
    return max(h2d_bytes / link["h2d_GBps"], d2h_bytes / link["d2h_GBps"],
               (h2d_bytes + d2h_bytes) / link["both_GBps"]) / 1e9


def measure_link(hx, dx, dy, dev, reps=5):
    """Copy-engine rates of the host link with the e2e run's own pinned buffer:
    host -> device, device -> host, and both at once on two streams (each a
    median of `reps` copies of hx's size, after two untimed)."""
    import torch
    hy = torch.empty_like(hx).pin_memory()
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    nb = hx.numel() * 4

    def timed(fn):
        for _ in range(2):
            fn()
        torch.cuda.synchronize(dev)
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s1)
            fn()
            e1.record(s1)
            torch.cuda.synchronize(dev)
            ts.append(e0.elapsed_time(e1) * 1e-3)
        return statistics.median(ts)

    def h2d():
        with torch.cuda.stream(s1):
            dx.copy_(hx, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s1):
            hy.copy_(dy, non_blocking=True)

    def both():
        ev = torch.cuda.Event()
        ev.record(s1)
        s2.wait_event(ev)
        with torch.cuda.stream(s2):
            hy.copy_(dy, non_blocking=True)
        with torch.cuda.stream(s1):
            dx.copy_(hx, non_blocking=True)
        s1.wait_stream(s2)

    th, td, tb = timed(h2d), timed(d2h), timed(both)
    del hy
    return {"h2d_GBps": round(nb / th / 1e9, 1), "d2h_GBps": round(nb / td / 1e9, 1),
            "both_GBps": round(2 * nb / tb / 1e9, 1), "bytes_per_copy": nb,
            "how": "pinned host <-> device copies of X's size on the copy engines, timed in this run"}


# --------------------------------------------------------------------- per-config block
# Every workload the targets are stated on, each kernel on its own input,
# both paths where a config has two.  (key, config, workload, kernel, path,
# target fraction of the measured peak or None where the config is reported
# only; C1's >= 0.85 applies at sweep sizes >= 256 MiB, see --sweep.)
CONFIG_ENTRIES = [
    ("C1_affine_auto", "C1", "affine_1m", "affine", "auto", None),
    ("C1_affine_vec4", "C1", "affine_1m", "affine", "vec4", None),
    ("C2_scale2d_aligned", "C2", "scale_8192", "scale2d", "aligned", 0.85),
    ("C2_scale2d_ragged_vec", "C2", "scale_8192", "scale2d", "ragged_vec", None),
    ("C3_copy2d_ragged", "C3", "ragged_4100", "copy2d", "ragged", 0.75),
    ("C3_scale2d_ragged", "C3", "ragged_4100", "scale2d", "ragged", 0.75),
    ("C4_rowsum", "C4", "coalesce_4096", "rowsum", "vec", 0.85),
    ("C4_colsum_auto", "C4", "coalesce_4096", "colsum", "auto", 0.70),
    ("C4_colsum_staged", "C4", "coalesce_4096", "colsum", "staged", 0.70),
    ("C5_rowmax_masked", "C5", "rowmax_8192", "rowmax_masked", "neg_inf", None),
    # the floors C1, C3, C4 and C5 are read against, timed the same way in
    # the same run: a device-to-device cudaMemcpyAsync of the maps' bytes,
    # and the plain streaming read of what the reductions read
    ("C1_floor_memcpy", "C1", "affine_1m", "memcpy", "d2d", None),
    ("C3_floor_memcpy", "C3", "ragged_4100", "memcpy", "d2d", None),
    ("C4_floor_read", "C4", "coalesce_4096", "read_probe", "u4", None),
    ("C5_floor_read", "C5", "rowmax_8192", "read_probe", "u4", None),
    # the same read with every block's share fixed at launch: the floor of the
    # column sum's one-pass forms, which give each CTA a fixed band of rows
    ("C4_floor_fixed_share", "C4", "coalesce_4096", "read_probe_fixed", "b512", None),
]
FIXED_SHARE_FLOOR_OF = {"C4_colsum_auto": "C4_floor_fixed_share", "C4_colsum_staged": "C4_floor_fixed_share"}
FLOOR_OF = {"C1": "C1_floor_memcpy", "C3": "C3_floor_memcpy", "C4": "C4_floor_read", "C5": "C5_floor_read"}
AMORTIZED_BYTES = 512 << 20  # rotating copies of the inputs and outputs: 4x the L2


def config_kernel(tm, kern, path, w, x, dev):
    """One kernel of a config: (describe, out_elems, call(X, O, W, stream, pdl),
    algorithmic bytes, workspace elems, check(out_host) -> bool)."""
    import numpy as np
    import oracle
    if kern == "affine":
        n = x.size
        var = {"auto": tm.TM_VAR_AUTO, "vec4": tm.TM_VAR_VEC4}[path]
        want = oracle.affine(x).view(np.uint32)
        return ("tm_affine %s, n=%d" % (path.upper(), n), n,
                lambda X, O, W, s, pdl: tm.tm_affine(X, O, n, var | (tm.TM_PDL if pdl else 0), s),
                8 * n, 0, lambda o: np.array_equal(o.view(np.uint32), want))
    if kern == "memcpy":
        n = x.size
        want = x.reshape(-1).view(np.uint32)

        def copy(X, O, W, s, pdl):
            O.copy_(X, non_blocking=True)  # on torch's current stream: the timed stream, or the capture stream
        return ("cudaMemcpyAsync device to device, %d bytes (torch copy_)" % (4 * n), n, copy, 8 * n, 0,
                lambda o: bool(np.array_equal(o.view(np.uint32), want)))
    M, N = x.shape
    if kern in ("scale2d", "copy2d"):
        TM_, TN_ = w["TM"], w["TN"]
        fl = tm.TM_ALIGNED if path == "aligned" else 0
        if kern == "scale2d":
            want = np.empty(M * N, np.float32)
            oracle.scale2d(x, N, want, N, M, N, ALPHA)
            want = want.view(np.uint32)
            call = lambda X, O, W, s, pdl: tm.tm_scale2d(X, N, O, N, M, N, ALPHA, TM_, TN_,
                                                         fl | (tm.TM_PDL if pdl else 0), s)
        else:
            want = np.empty(M * N, np.uint32)
            oracle.copy2d(x, N, want, N, M, N)
            call = lambda X, O, W, s, pdl: tm.tm_copy2d(X, N, O, N, M, N, TM_, TN_, fl | (tm.TM_PDL if pdl else 0), s)
        how = "aligned promise (no masks, 32-byte vectors)" if fl else \
            "no promise: ragged path (16-byte vectors, one predicate each)"
        return ("tm_%s [%d,%d] %dx%d tiles, %s" % (kern, M, N, TM_, TN_, how), M * N, call, 8 * M * N, 0,
                lambda o: np.array_equal(o.view(np.uint32), want))
    absx = np.abs(x.astype(np.float64))
    if kern == "rowsum":
        want, tol = oracle.rowsum(x, N, M, N), 1e-5 * absx.sum(axis=1)
        return ("tm_rowsum [%d,%d] 2x512 tiles" % (M, N), M,
                lambda X, O, W, s, pdl: tm.tm_rowsum(X, N, M, N, O, 2, 512, tm.TM_PDL if pdl else 0, s),
                4 * M * N + 4 * M, 0, lambda o: bool(np.all(np.abs(o - want) <= tol)))
    if kern == "colsum":
        var = {"auto": tm.TM_VAR_AUTO, "staged": tm.TM_VAR_STAGED}[path]
        ws = tm.tm_colsum_workspace_bytes(M, N, 32, 128, var)
        want, tol = oracle.colsum(x, N, M, N), 1e-5 * absx.sum(axis=0)
        return ("tm_colsum %s [%d,%d] 32x128 (workspace %d B)" % (path.upper(), M, N, ws), N,
                lambda X, O, W, s, pdl: tm.tm_colsum(X, N, M, N, O, W, ws, 32, 128, var, tm.TM_PDL if pdl else 0, s),
                4 * M * N + 4 * N, max(ws // 4, 4), lambda o: bool(np.all(np.abs(o - want) <= tol)))
    if kern == "read_probe":
        n = M * N
        U = int(path[1:])
        blocks = tm.tm_read_probe_blocks(n, U)
        span = 1024 * U  # block b sums elements [b*span, (b+1)*span) of the flat tensor
        xb = np.zeros(blocks * span, np.float32)
        xb[:n] = x.reshape(-1)
        xb = xb.reshape(blocks, span)
        want = oracle.rowsum(xb, span, blocks, span)
        tol = 1e-5 * np.abs(xb.astype(np.float64)).sum(axis=1)
        return ("tm_read_probe, %d floats, %d 16-byte loads per thread (no TM_PDL: plain launches)" % (n, U), blocks,
                lambda X, O, W, s, pdl: tm.tm_read_probe(X, n, O, U, s), 4 * n + 4 * blocks, 0,
                lambda o: bool(np.all(np.abs(o - want) <= tol)))
    if kern == "read_probe_fixed":
        n = M * N
        blocks = int(path[1:])
        share = tm.tm_read_probe_fixed_share(n, blocks)
        xb = np.zeros(blocks * share, np.float32)
        xb[:n] = x.reshape(-1)
        xb = xb.reshape(blocks, share)
        want = oracle.rowsum(xb, share, blocks, share)
        tol = 1e-5 * np.abs(xb.astype(np.float64)).sum(axis=1)
        return ("tm_read_probe_fixed, %d floats, %d blocks of fixed %d-float shares (plain launches)"
                % (n, blocks, share), blocks,
                lambda X, O, W, s, pdl: tm.tm_read_probe_fixed(X, n, O, blocks, s), 4 * n + 4 * blocks, 0,
                lambda o: bool(np.all(np.abs(o - want) <= tol)))
    if kern == "rowmax_masked":
        BC = w["BC"]
        want = oracle.rowmax_masked(x, N, M, N, BC)
        return ("tm_rowmax_masked [%d,%d] 8 rows x %d-column tiles, -inf fill (where/iota remainder tile of %d)"
                % (M, N, BC, N % BC), M,
                lambda X, O, W, s, pdl: tm.tm_rowmax_masked(X, N, M, N, O, 8, BC, tm.TM_FILL_NEG_INF,
                                                            tm.TM_PDL if pdl else 0, s),
                4 * M * N + 4 * M, 0, lambda o: bool(np.array_equal(o, want) and np.all(o < 0)))
    raise ValueError(kern)


def run_configs(tm, dev, peak, reps=20, verify=True, x_step=None):
    """Each entry of CONFIG_ENTRIES two ways: a lone launch after an L2 flush
    (median of `reps`), and back-to-back overlapped launches (TM_PDL) captured
    in one CUDA graph, over rotating copies of the input and output that
    together exceed 4x the L2, so neither side is served from L2.  Every
    output is checked against the oracle before it is timed (and the last
    copy written again after the back-to-back run)."""
    import torch

    from masking_tm_affine_gb300 import synth
    out = {}
    flush = L2Flush(dev, "dirty")
    flush_clean = L2Flush(dev, "clean")
    inputs = {}

    def lone_times(fl, call, X, O, W, stream, s):
        ts = []
        for rep in range(reps + 3):
            fl()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call(X, O, W, s, False)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            if rep >= 3:
                ts.append(e0.elapsed_time(e1) * 1e-3)
        return statistics.median(ts), statistics.fmean(ts)
    for key, cfg, wl, kern, path, target in CONFIG_ENTRIES:
        if wl not in inputs:
            inputs[wl] = x_step if (wl == WORKLOAD and x_step is not None) else synth.workload_input(wl)
        x = inputs[wl]
        w = synth.WORKLOADS[wl]
        desc, on, call, nbytes, wn, check = config_kernel(tm, kern, path, w, x, dev)
        X0 = torch.from_numpy(x.reshape(-1)).to(dev)
        in_out = X0.numel() * 4 + on * 4
        R = max(1, -(-AMORTIZED_BYTES // in_out))
        Xs = [X0] + [X0.clone() for _ in range(R - 1)]
        Os = [torch.full((on,), float("nan"), dtype=torch.float32, device=dev) for _ in range(R)]
        W = torch.empty(max(wn, 4), dtype=torch.float32, device=dev)
        stream = torch.cuda.current_stream(dev)
        s = stream.cuda_stream
        call(Xs[0], Os[0], W, s, False)
        tm.tm_check(s)
        ok = check(Os[0].cpu().numpy()) if verify else None
        if verify and not ok:
            raise AssertionError("%s: output differs from the oracle" % key)
        # lone launches, L2 flushed before each: the flush's lines left dirty
        # (the launch pays their write-back), and cleaned by a read after it
        lone, lone_mean = lone_times(flush, call, Xs[0], Os[0], W, stream, s)
        lone_c, lone_c_mean = lone_times(flush_clean, call, Xs[0], Os[0], W, stream, s)
        # back to back: n overlapped calls in one graph, rotating over R copies
        n = max(100, min(1000, int(2e-3 / max(lone_mean, 1e-6)) + 1))
        n = -(-n // R) * R
        side = torch.cuda.Stream(device=dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            call(Xs[0], Os[0], W, side.cuda_stream, False)  # warm the call path on the capture stream
        torch.cuda.synchronize(dev)
        with torch.cuda.graph(g, stream=side):
            cs = side.cuda_stream
            for i in range(n):
                call(Xs[i % R], Os[i % R], W, cs, True)
        ts = []
        for rep in range(5):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            if rep >= 2:
                ts.append(e0.elapsed_time(e1) * 1e-3 / n)
        tm.tm_check(s)
        amort = statistics.median(ts)
        if verify and not check(Os[(n - 1) % R].cpu().numpy()):
            raise AssertionError("%s: back-to-back output differs from the oracle" % key)
        row = {"config": cfg, "workload": wl, "kernel": desc, "bytes": nbytes,
               "lone": {"us": round(lone * 1e6, 2), "us_mean": round(lone_mean * 1e6, 2),
                        "GBps": round(gbps(nbytes, lone), 1), "frac": round(gbps(nbytes, lone) / peak, 4),
                        "reps": reps, "l2": "512 MiB dirty flush before each launch"},
               "lone_clean": {"us": round(lone_c * 1e6, 2), "us_mean": round(lone_c_mean * 1e6, 2),
                              "GBps": round(gbps(nbytes, lone_c), 1), "frac": round(gbps(nbytes, lone_c) / peak, 4),
                              "reps": reps, "l2": "512 MiB write then 256 MiB read before each launch: "
                                                  "cold L2 of clean lines, as under ncu"},
               "back_to_back": {"us_per_call": round(amort * 1e6, 3), "GBps": round(gbps(nbytes, amort), 1),
                                "frac": round(gbps(nbytes, amort) / peak, 4), "calls": n, "copies": R,
                                "how": "TM_PDL calls in one CUDA graph; inputs and outputs rotate over the copies "
                                       "(%d MiB in all), so none is read from L2" % (R * in_out >> 20)},
               "target": target, "verified": ok}
        if target is not None:
            row["target_met"] = {"lone": row["lone"]["frac"] >= target,
                                 "lone_clean": row["lone_clean"]["frac"] >= target,
                                 "back_to_back": row["back_to_back"]["frac"] >= target}
        out[key] = row
        del Xs, Os, W, X0, g
        torch.cuda.empty_cache()
    attach_floors(out)
    return out


def attach_floors(rows):
    """Each row of the configs block against its config's floor row
    (FLOOR_OF), timed the same way in the same run: its lone times over the
    floor's, and for a targeted row whether the dirty-flush lone time is
    within 5 % of it."""
    floors = set(FLOOR_OF.values()) | set(FIXED_SHARE_FLOOR_OF.values())
    for key, row in rows.items():
        ff = FIXED_SHARE_FLOOR_OF.get(key)
        if ff in rows:
            f = rows[ff]
            row["floor_fixed_share"] = {"entry": ff, "lone_vs_floor": round(row["lone"]["us"] / f["lone"]["us"], 3),
                                        "lone_clean_vs_floor": round(row["lone_clean"]["us"] / f["lone_clean"]["us"], 3)}
        fk = FLOOR_OF.get(row["config"])
        if fk not in rows or key in floors:
            continue
        f = rows[fk]
        row["floor"] = {"entry": fk,
                        "lone_frac": f["lone"]["frac"], "lone_clean_frac": f["lone_clean"]["frac"],
                        "lone_vs_floor": round(row["lone"]["us"] / f["lone"]["us"], 3),
                        "lone_clean_vs_floor": round(row["lone_clean"]["us"] / f["lone_clean"]["us"], 3),
                        "how": "this row's lone time over the floor's (1.0 = as fast as the floor; "
                               "both move the same input bytes)"}
        if row["target"] is not None:
            row["target_met"]["lone_within_5pct_of_floor"] = row["lone"]["us"] <= 1.05 * f["lone"]["us"]
    return rows


# --------------------------------------------------------------------- reference arm
def run_reference(args):
    """The CPU oracle as the reference arm: same metric and workload, each step
    one pass over a row slice sized so the whole run stays within minutes."""
    import numpy as np
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    import oracle
    from masking_tm_affine_gb300 import synth
    oracle.build()
    x = synth.workload_input(WORKLOAD)
    prev = os.sched_getaffinity(0) if hasattr(os, "sched_getaffinity") else None
    if prev:
        os.sched_setaffinity(0, {min(prev)})

    Yall = np.empty_like(x)
    Ball = np.empty(x.size, dtype=np.uint32)

    def one_pass(R):
        xs = x[:R]
        Yw = Yall[:R]
        Bw = Ball[:R * N]
        oracle.affine(xs)
        oracle.scale2d(xs, N, Yw, N, R, N, ALPHA)
        oracle.copy2d(xs, N, Bw, N, R, N)
        oracle.rowsum(xs, N, R, N)
        oracle.colsum(xs, N, R, N)
        oracle.rowmax_masked(xs, N, R, N, 64)

    t0 = time.perf_counter()
    one_pass(64)
    per_row = (time.perf_counter() - t0) / 64
    budget = 90.0
    R = int(max(1, min(M, budget / max(args.steps + args.warmup, 1) / per_row)))
    for _ in range(args.warmup):
        one_pass(R)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one_pass(R)
    el = time.perf_counter() - t0
    if prev:
        os.sched_setaffinity(0, prev)
    by = sum(kernel_bytes(R, N).values()) * args.steps
    v = round(gbps(by, el), 3)
    sample = ("oracle step (all six maps) over rows [0,%d) of the [8192,8192] batch per step, single thread "
              "pinned to one core of %d" % (R, os.cpu_count()))
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic: numpy PCG64, X ~ N(0,1) seed 1, rounded once to fp32",
            "config": {"workload": "scale_8192 (row slice per step, see cpu_baseline.sample)", "M": R, "N": N},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# --------------------------------------------------------------------- L2 flush
class L2Flush:
    """Evicts L2 between timed launches with a 512 MiB write (larger than the
    126 MB L2).  mode "dirty" stops there: the timed launch first writes back
    the flush's dirty lines as it fills L2 (pessimistic for short kernels).
    mode "clean" then reads 256 MiB of another buffer, so the launch starts
    from a cold L2 of clean lines, as under ncu's cache control; a kernel with
    outputs may then leave up to an L2 of them dirty at its end, written back
    after the timed region (optimistic for maps under ~256 MiB)."""

    def __init__(self, dev, mode="dirty"):
        import torch
        self.mode = mode
        self.w = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
        self.r = torch.zeros(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev) if mode == "clean" else None

    def __call__(self):
        self.w.zero_()
        if self.r is not None:
            self.r.sum()

    @property
    def note(self):
        if self.mode == "clean":
            return "flushed before each launch (512 MiB write, then 256 MiB read: cold, clean L2)"
        return "flushed before each launch (512 MiB write: cold L2 full of the flush's dirty lines)"


# --------------------------------------------------------------------- size sweep
def run_sweep(args):
    """Y = 1.5*X over tensors of 2^10 .. 2^30 bytes (and the affine map over the
    same sizes, AUTO and VEC4), median of CUDA-event times with L2 flushed
    between reps."""
    import torch

    from masking_tm_affine_gb300 import tm
    tm.load()
    dev = torch.device("cuda", 0)
    peak, _ = measured_peak()
    flush = L2Flush(dev, args.flush)
    stream = torch.cuda.current_stream(dev)
    out = []
    lo, hi = (int(v) for v in args.sweep_lg.split("-"))
    for lg in range(lo, hi + 1):
        E = (1 << lg) // 4
        if E >= 4096:
            n = min(8192, E // 32)
            shape, flags = (E // n, n), tm.TM_ALIGNED
        else:
            shape, flags = (1, E), 0
        X = torch.randn(E, device=dev, generator=torch.Generator(device=dev).manual_seed(lg))  # values are immaterial
        Y = torch.empty_like(X)
        A1 = torch.empty_like(X)
        res = {}
        for name, fn in (("scale2d", lambda: tm.tm_scale2d(X, shape[1], Y, shape[1], shape[0], shape[1], ALPHA,
                                                          32, 128, flags, stream.cuda_stream)),
                         ("affine", lambda: tm.tm_affine(X, A1, E, tm.TM_VAR_AUTO, stream.cuda_stream)),
                         ("affine_vec4", lambda: tm.tm_affine(X, A1, E, tm.TM_VAR_VEC4, stream.cuda_stream))):
            ts = []
            for rep in range(args.sweep_reps + 3):
                flush()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                torch.cuda.synchronize(dev)
                if rep >= 3:
                    ts.append(e0.elapsed_time(e1) * 1e-3)
            t = statistics.median(ts)
            res[name] = {"us": round(t * 1e6, 2), "GBps": round(gbps(8 * E, t), 1), "frac": round(gbps(8 * E, t) / peak, 4)}
        out.append({"bytes_per_tensor": 1 << lg, "shape": list(shape), **res, "l2": flush.note})
        del X, Y, A1
    tm.tm_check()
    return out


# --------------------------------------------------------------------- single-workload cases
CASES = {
    # name: (workload, kernel, variants) -- variants[0] is the default
    "affine_1m": ("affine_1m", "affine", ["auto", "scalar", "vec_unaligned", "vec4", "vec8"]),
    "scale_8192": ("scale_8192", "scale2d", ["aligned", "ragged_vec", "scalar"]),
    "ragged_copy": ("ragged_4100", "copy2d", ["auto", "scalar"]),
    "ragged_scale": ("ragged_4100", "scale2d", ["auto", "scalar"]),
    "aligned_copy": ("aligned_4096", "copy2d", ["aligned", "auto"]),
    "rowsum_4096": ("coalesce_4096", "rowsum", ["vec", "scalar"]),
    "colsum_4096": ("coalesce_4096", "colsum", ["auto", "staged", "regdirect", "naive", "cluster"]),
    # the plain streaming read of the same 64 MiB: the floor the sums are compared with
    "read_floor_4096": ("coalesce_4096", "read_probe", ["u4", "u1", "u2", "u8", "u16"]),
    "rowmax_8192": ("rowmax_8192", "rowmax_masked", ["neg_inf", "zero", "scalar"]),
    "softmax_8192": ("rowmax_8192", "softmax_rowstats", ["neg_inf", "zero", "scalar"]),
    "pad_ragged": ("ragged_4100", "pad2d", ["auto"]),
    "channel_nhwc": ("channel_nhwc", "channel_affine", ["auto", "scalar"]),
    "channel_nchw": ("channel_nchw", "channel_affine", ["auto", "scalar"]),
    # the reductions on the [8192, 8192] batch of the step, for tile tuning
    "softmax_8192sq": ("scale_8192", "softmax_rowstats", ["neg_inf"]),
    "rowsum_8192sq": ("scale_8192", "rowsum", ["vec"]),
    "colsum_8192sq": ("scale_8192", "colsum", ["auto", "staged", "regdirect", "cluster"]),
    "rowmax_8192sq": ("scale_8192", "rowmax_masked", ["neg_inf"]),
    "read_floor_8192sq": ("scale_8192", "read_probe", ["u4", "u8"]),
    # the same reads with every block's share fixed at launch (512 / 608 blocks):
    # the floor of a one-pass walk that cannot rebalance, like the column sums'
    "read_fixed_4096": ("coalesce_4096", "read_probe_fixed", ["b512", "b608"]),
    "read_fixed_8192sq": ("scale_8192", "read_probe_fixed", ["b512", "b608"]),
    # the tensor-core gemm (3xTF32 by default; tf32 = one pass)
    "gemm_4100": ("gemm_4100", "gemm", ["3xtf32", "tf32"]),
    "gemm_8192": ("gemm_8192", "gemm", ["3xtf32", "tf32"]),
}

# nominal tf32 / bf16 dense tensor rates of GB300 (1.1 and 2.25 PFLOP/s): the
# tf32 peak is the measured bf16 peak times this ratio
TF32_PER_BF16 = 1.1 / 2.25


def tf32_peak(sustained: bool = False):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    try:
        with open(path) as f:
            v = float(json.load(f)[key])
        return v * TF32_PER_BF16, "measured (MEASURED_PEAKS.json %s x 1.1/2.25 nominal tf32/bf16)" % key
    except Exception:
        return 1900.0 * TF32_PER_BF16, "fallback (1.9 PFLOP/s bf16 x 1.1/2.25)"


def time_oracle_gemm(w, a, b, c, budget_s: float = 1.5) -> dict:
    """The oracle's row-by-row fp64 gemm on one host thread, rows sized to about budget_s."""
    import numpy as np
    import oracle
    oracle.build()
    M, N, K = w["M"], w["N"], w["K"]
    t0 = time.perf_counter()
    oracle.gemm_rows(a, K, b, N, c, N, np.arange(1), N, K, w["alpha"], w["beta"])
    per = time.perf_counter() - t0
    R = int(max(1, min(M, budget_s / max(per, 1e-9))))
    t0 = time.perf_counter()
    oracle.gemm_rows(a, K, b, N, c, N, np.arange(R), N, K, w["alpha"], w["beta"])
    el = time.perf_counter() - t0
    return {"TFLOPs": round(2.0 * R * N * K / el / 1e12, 6), "sample": "%d of %d rows, one host thread" % (R, M)}


def run_gemm_case(name, args, dev, stream, flush):
    import torch

    from masking_tm_affine_gb300 import synth, tm
    wl, _, variants = CASES[name]
    w = synth.WORKLOADS[wl]
    M, N, K = w["M"], w["N"], w["K"]
    a, b, c = synth.gemm_inputs(wl)
    A, B = torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev)
    C0 = torch.from_numpy(c).to(dev)
    C = C0.clone()
    parts = [int(t) for t in args.tile.split("x")] if args.tile else []
    TM_ = parts[0] if parts else w["TM"]
    TN_ = parts[1] if len(parts) > 1 else w["TN"]
    TK_ = parts[2] if len(parts) > 2 else w["TK"]
    wsb = tm.tm_gemm_workspace_bytes(M, N, K, TN_)
    raw = torch.empty(wsb + 1024, dtype=torch.uint8, device=dev)
    ws = (raw.data_ptr() + 1023) // 1024 * 1024
    aligned = M % TM_ == 0 and N % TN_ == 0 and K % TK_ == 0
    peak, peak_src = tf32_peak()
    s = stream.cuda_stream
    out = []
    chosen = variants if args.variant == "all" else [args.variant or variants[0]]
    for v in chosen:
        fl = (tm.TM_ALIGNED if aligned else 0) | (tm.TM_GEMM_TF32 if v == "tf32" else 0)
        ts = []
        for rep in range(args.reps + 3):
            C.copy_(C0)
            if not args.no_flush:
                flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            tm.tm_gemm(A, K, B, N, C, N, M, N, K, w["alpha"], w["beta"], ws, wsb, TM_, TN_, TK_, fl, s)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            if rep >= 3:
                ts.append(e0.elapsed_time(e1) * 1e-3)
        t = statistics.median(ts)
        flops = 2.0 * M * N * K
        passes = 3 if v == "3xtf32" else 1
        row = {"case": name, "kernel": "gemm", "variant": v, "tile": "%dx%dx%d" % (TM_, TN_, TK_), "M": M, "N": N, "K": K,
               "us": round(t * 1e6, 2), "TFLOPs": round(flops / t / 1e12, 2),
               "tensor_TFLOPs": round(passes * flops / t / 1e12, 2),
               "frac_of_tf32_peak": round(passes * flops / t / 1e12 / peak, 4), "tf32_peak": round(peak, 1),
               "peak_source": peak_src, "reps": args.reps,
               "l2": flush.note if not args.no_flush else "warm"}
        if args.oracle:
            row["oracle"] = time_oracle_gemm(w, a, b, c)
        out.append(row)
    # context: cuBLAS through torch.matmul on the same operands, fp32 and tf32
    # math (C = alpha A B + beta C via addmm), same flush and event timing
    for label, tf32 in (("cublas_fp32", False), ("cublas_tf32", True)):
        prev = torch.backends.cuda.matmul.allow_tf32
        torch.backends.cuda.matmul.allow_tf32 = tf32
        ts = []
        for rep in range(min(args.reps, 10) + 3):
            C.copy_(C0)
            if not args.no_flush:
                flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            torch.addmm(C, A, B, beta=w["beta"], alpha=w["alpha"], out=C)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            if rep >= 3:
                ts.append(e0.elapsed_time(e1) * 1e-3)
        torch.backends.cuda.matmul.allow_tf32 = prev
        t = statistics.median(ts)
        out.append({"case": name, "kernel": label, "us": round(t * 1e6, 2),
                    "TFLOPs": round(2.0 * M * N * K / t / 1e12, 2), "note": "library reference, context only"})
    return out


def time_oracle_case(kern, w, x, budget_s: float = 1.5) -> dict:
    """The oracle on one host core for the same kernel and workload, over a row
    slice sized to about budget_s (whole workload when it fits)."""
    import numpy as np
    import oracle
    from masking_tm_affine_gb300 import synth
    oracle.build()
    flat = kern == "affine"
    rows = x.size if flat else x.shape[0]
    cols = 1 if flat else x.shape[1]

    def call(R):
        if flat:
            oracle.affine(x[:R])
            return 8 * R
        xs = np.ascontiguousarray(x[:R])
        if kern in ("scale2d", "copy2d"):
            Y = np.empty(R * cols, dtype=np.float32)
            if kern == "scale2d":
                oracle.scale2d(xs, cols, Y, cols, R, cols, ALPHA)
            else:
                oracle.copy2d(xs, cols, Y.view(np.uint32), cols, R, cols)
            return 8 * R * cols
        if kern == "rowsum":
            oracle.rowsum(xs, cols, R, cols)
            return 4 * R * cols + 4 * R
        if kern in ("read_probe", "read_probe_fixed"):  # a plain read of the same bytes: the oracle's row sums
            oracle.rowsum(xs, cols, R, cols)
            return 4 * R * cols
        if kern == "colsum":
            oracle.colsum(xs, cols, R, cols)
            return 4 * R * cols + 4 * cols
        if kern == "rowmax_masked":
            oracle.rowmax_masked(xs, cols, R, cols, w.get("BC", 64))
            return 4 * R * cols + 4 * R
        if kern == "softmax_rowstats":
            oracle.softmax_rowstats(xs, cols, R, cols, w.get("BC", 64))
            return 4 * R * cols + 8 * R
        if kern == "channel_affine":
            sc, bi = synth.channel_params(w["C"])
            Y = np.empty(R * cols, dtype=np.float32)
            oracle.channel_affine(xs, cols, R, cols, sc, bi, w["C"], w["layout"], Y, cols)
            return 8 * R * cols + 8 * w["C"]
        if kern == "pad2d":
            Np = -(-cols // w["TN"]) * w["TN"]
            Rp = -(-R // w["TM"]) * w["TM"]
            B = np.empty(Rp * Np, dtype=np.uint32)
            oracle.pad2d(xs, cols, R, cols, B, Np, Rp, Np)
            return 4 * R * cols + 4 * Rp * Np
        raise ValueError(kern)

    probe = max(1, min(rows, 64 if not flat else 1 << 16))
    t0 = time.perf_counter()
    call(probe)
    per = (time.perf_counter() - t0) / probe
    R = int(max(1, min(rows, budget_s / max(per, 1e-12))))
    t0 = time.perf_counter()
    nb = call(R)
    el = time.perf_counter() - t0
    return {"GBps": round(gbps(nb, el), 3), "sample": "%d of %d %s, one host thread" % (R, rows, "elements" if flat else "rows")}


def run_cases(args):
    """Time one kernel on one workload: median of CUDA-event times over
    --reps launches, L2 flushed (L2Flush) before every launch."""
    import torch

    from masking_tm_affine_gb300 import synth, tm
    tm.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, _ = measured_peak()
    stream = torch.cuda.current_stream(dev)
    s = stream.cuda_stream
    flush = L2Flush(dev, args.flush)
    names = list(CASES) if args.case == "all" else [args.case]
    out = []
    for name in names:
        wl, kern, variants = CASES[name]
        if kern == "gemm":
            out.extend(run_gemm_case(name, args, dev, stream, flush))
            continue
        w = synth.WORKLOADS[wl]
        x = synth.workload_input(wl)
        X = torch.from_numpy(x.reshape(-1)).to(dev)
        if kern == "affine":
            n = x.size
            O = torch.empty_like(X)
            vmap = {"auto": tm.TM_VAR_AUTO, "scalar": tm.TM_VAR_SCALAR, "vec_unaligned": tm.TM_VAR_VEC_UNALIGNED,
                    "vec4": tm.TM_VAR_VEC4, "vec8": tm.TM_VAR_VEC8}
            nbytes = 8 * n
            mk = lambda v: (lambda: tm.tm_affine(X, O, n, vmap[v], s))
        else:
            Mw, Nw = w["M"], w["N"]
            tile = tuple(int(t) for t in args.tile.split("x")) if args.tile else None
            if kern in ("scale2d", "copy2d"):
                O = torch.empty_like(X)
                nbytes = 8 * Mw * Nw
                TM_, TN_ = tile or (w["TM"], w["TN"])
                fl = {"aligned": tm.TM_ALIGNED, "ragged_vec": 0, "auto": 0, "scalar": tm.TM_PATH_SCALAR}
                if kern == "scale2d":
                    mk = lambda v: (lambda: tm.tm_scale2d(X, Nw, O, Nw, Mw, Nw, ALPHA, TM_, TN_, fl[v], s))
                else:
                    mk = lambda v: (lambda: tm.tm_copy2d(X, Nw, O, Nw, Mw, Nw, TM_, TN_, fl[v], s))
            elif kern == "rowsum":
                O = torch.empty(Mw, dtype=torch.float32, device=dev)
                nbytes = 4 * Mw * Nw + 4 * Mw
                fl = {"vec": 0, "scalar": tm.TM_PATH_SCALAR}
                # [4096, 4096]: 2 rows x 512 columns per block fills one wave (ncu sweep:
                # 12.6 us vs 13.4 us at 1 x 1024); the step's [8192, 8192] keeps ROWSUM_TILE
                RT_, RN_ = tile or ((2, 512) if Mw * Nw <= (1 << 24) else ROWSUM_TILE)
                mk = lambda v: (lambda: tm.tm_rowsum(X, Nw, Mw, Nw, O, RT_, RN_, fl[v], s))
            elif kern == "colsum":
                O = torch.empty(Nw, dtype=torch.float32, device=dev)
                nbytes = 4 * Mw * Nw + 4 * Nw
                vm = {"auto": tm.TM_VAR_AUTO, "staged": tm.TM_VAR_STAGED, "regdirect": tm.TM_VAR_REGDIRECT,
                      "cluster": tm.TM_VAR_CLUSTER,
                      "naive": tm.TM_VAR_NAIVE}
                CT_, CN_ = tile or COLSUM_TILE
                ws = max(tm.tm_colsum_workspace_bytes(Mw, Nw, CT_, CN_, tm.TM_VAR_NAIVE),
                         tm.tm_colsum_workspace_bytes(Mw, Nw, CT_, CN_, tm.TM_VAR_AUTO))
                Wt = torch.empty(ws // 4, dtype=torch.float32, device=dev)
                mk = lambda v: (lambda: tm.tm_colsum(X, Nw, Mw, Nw, O, Wt, ws, CT_, CN_, vm[v], 0, s))
            elif kern == "read_probe":
                U = {"u1": 1, "u2": 2, "u4": 4, "u8": 8, "u16": 16}
                O = torch.empty(max(tm.tm_read_probe_blocks(Mw * Nw, 1), 1), dtype=torch.float32, device=dev)
                nbytes = 4 * Mw * Nw
                mk = lambda v: (lambda: tm.tm_read_probe(X, Mw * Nw, O, U[v], s))
            elif kern == "read_probe_fixed":
                O = torch.empty(65535, dtype=torch.float32, device=dev)
                nbytes = 4 * Mw * Nw
                mk = lambda v: (lambda: tm.tm_read_probe_fixed(X, Mw * Nw, O, int(v[1:]), s))
            elif kern == "pad2d":
                Mp_, Np_ = tm.tm_padded_extent(Mw, [w["TM"]]), tm.tm_padded_extent(Nw, [w["TN"]])
                ldp = tm.tm_row_stride(Np_, 16)
                O = torch.empty(Mp_ * ldp, dtype=torch.float32, device=dev)
                nbytes = 4 * Mw * Nw + 4 * Mp_ * Np_
                mk = lambda v: (lambda: tm.tm_pad2d(X, Nw, Mw, Nw, O, ldp, Mp_, Np_, s))
            elif kern == "channel_affine":
                O = torch.empty_like(X)
                nbytes = 8 * Mw * Nw + 8 * w["C"]
                scv, biv = synth.channel_params(w["C"])
                SC = torch.from_numpy(scv).to(dev)
                BI = torch.from_numpy(biv).to(dev)
                TM_, TN_ = tile or (w["TM"], w["TN"])
                fl = {"auto": 0, "scalar": tm.TM_PATH_SCALAR}
                mk = lambda v: (lambda: tm.tm_channel_affine(X, Nw, Mw, Nw, SC, BI, w["C"], w["layout"], O, Nw,
                                                             TM_, TN_, fl[v], s))
            elif kern == "softmax_rowstats":
                O = torch.empty(Mw, dtype=torch.float32, device=dev)
                O2 = torch.empty(Mw, dtype=torch.float32, device=dev)
                nbytes = 4 * Mw * Nw + 8 * Mw
                fm = {"neg_inf": (tm.TM_FILL_NEG_INF, 0), "zero": (tm.TM_FILL_ZERO, 0),
                      "scalar": (tm.TM_FILL_NEG_INF, tm.TM_PATH_SCALAR)}
                SB_, SC_ = tile or (16 if Nw < 4096 else 8, w.get("BC", 64))  # wide rows: a warp per row
                mk = lambda v: (lambda: tm.tm_softmax_rowstats(X, Nw, Mw, Nw, O, O2, SB_, SC_, fm[v][0], fm[v][1], s))
            else:
                O = torch.empty(Mw, dtype=torch.float32, device=dev)
                nbytes = 4 * Mw * Nw + 4 * Mw
                fm = {"neg_inf": (tm.TM_FILL_NEG_INF, 0), "zero": (tm.TM_FILL_ZERO, 0),
                      "scalar": (tm.TM_FILL_NEG_INF, tm.TM_PATH_SCALAR)}
                BR_, BC_ = tile or (8 if Nw < 4096 else ROWMAX_BR, w.get("BC", 64))  # short rows: 8 per block
                mk = lambda v: (lambda: tm.tm_rowmax_masked(X, Nw, Mw, Nw, O, BR_, BC_, fm[v][0], fm[v][1], s))
        chosen = variants if args.variant == "all" else [args.variant or variants[0]]
        for v in chosen:
            fn = mk(v)
            ts = []
            for rep in range(args.reps + 3):
                if not args.no_flush:
                    flush()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                torch.cuda.synchronize(dev)
                if rep >= 3:
                    ts.append(e0.elapsed_time(e1) * 1e-3)
            t = statistics.median(ts)
            tmean = statistics.fmean(ts)  # events tick in ~2 us steps: the mean resolves short kernels better
            row = {"case": name, "kernel": kern, "variant": v, "tile": args.tile, "bytes": nbytes, "us": round(t * 1e6, 2),
                   "GBps": round(gbps(nbytes, t), 1), "frac": round(gbps(nbytes, t) / peak, 4),
                   "us_mean": round(tmean * 1e6, 2), "GBps_mean": round(gbps(nbytes, tmean), 1),
                   "reps": args.reps, "l2": flush.note if not args.no_flush else "warm"}
            if args.oracle:
                row["oracle"] = time_oracle_case(kern, w, x)
            out.append(row)
        del X, O
    tm.tm_check()
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sweep", action="store_true", help="print the 1 KB..1 GB size sweep instead")
    ap.add_argument("--sweep-reps", type=int, default=20)
    ap.add_argument("--sweep-lg", default="10-30", help="--sweep: log2 byte sizes per tensor, LO-HI")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--e2e-mode", choices=["pipelined", "serial"], default="pipelined")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-verify", action="store_true")
    ap.add_argument("--case", help="time one kernel on one workload instead (%s, or all)" % ", ".join(CASES))
    ap.add_argument("--variant", help="variant of --case (default: the first; 'all' for every one)")
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--tile", help="--case: tile override, e.g. 1x1024 (rows x columns)")
    ap.add_argument("--no-flush", action="store_true", help="--case: do not flush L2 between launches")
    ap.add_argument("--flush", choices=["dirty", "clean"], default="dirty",
                    help="--case/--sweep: leave the flush's lines dirty (default) or clean (see L2Flush)")
    ap.add_argument("--oracle", action="store_true", help="--case: also time the oracle on the same workload")
    ap.add_argument("--min-timed-s", type=float, default=1.0,
                    help="repeat the K-step timed region until this many seconds have passed (at least 3 times)")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-config block")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    if args.case:
        for row in run_cases(args):
            print(json.dumps(row))
        return
    if args.impl == "reference":
        line = run_reference(args)
    elif args.sweep:
        for row in run_sweep(args):
            print(json.dumps(row))
        return
    else:
        line = run_gpu(args)
    if line is not None:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
