"""Throughput of the fused add + Gemma RMSNorm + quant op on GB300.

One step = one call of the op over one batch of the largest workload (prefill,
M=16384, H=8192, fp16, static FP8 with an in-place residual: 939.5 MB per
call); the per-workload table adds the decode, M=2048 and
tensor-parallel-partial shapes and the method's variants.  Prints ONE JSON
line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gnq|reference]

Timing: W untimed steps, then exactly K steps captured in one CUDA graph and
timed with CUDA events on the capture stream, bracketed by a barrier and a
device synchronize.  Steps rotate over at least eight input/output sets;
each step's inputs are larger than L2 and the sets together exceed twice
the L2 size, so no step finds its inputs in L2.  Under
torchrun every rank runs an independent replica (rows are independent, there
is no data exchange); the slowest rank's time is reported and the value is
the bytes all ranks moved over that time.

--impl reference times the CPU oracle (the plain C restatement of the method)
on the same workload, metric and unit, on this machine's host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from nvfp4_quant_gemma_gb300.workloads import (HEADLINE, SMALL_M, SWEEP_BASES,  # noqa: E402
                                                WORKLOADS, DTYPES, all_workloads, make_inputs,
                                                sweep_workload)

METRIC = "achieved HBM GB/s (% of GB300 peak) and tokens/s for add+GemmaRMSNorm+quant"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["nvfp4_quant_gemma_gb300/csrc/" + f for f in (
    "gnq_device.cuh", "gnq_kernels.cuh", "gnq_launch.cuh", "gnq_api.cu", "gnq_mode_none.cu",
    "gnq_mode_fp8.cu", "gnq_mode_nvfp4.cu", "gnq_mode_mxfp8.cu")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------

def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    try:
        lines = open(TRAFFIC_FILE).read().splitlines()
    except OSError:
        return None
    src_hash = None
    table = {}
    for ln in lines:
        ln = ln.strip()
        if not ln or ln.startswith("#"):
            continue
        parts = ln.split()
        if parts[0] == "kernel_sources_sha256_16":
            src_hash = parts[1]
        elif len(parts) >= 2:
            table[parts[0]] = parts[1]
    if src_hash != kernel_hash() or workload not in table:
        return None
    v = table[workload]
    return None if v == "null" else float(v)


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons over a window."""

    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        rows = []
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 10:
                continue
            if self.uuid and f[1] != self.uuid:
                continue
            rows.append(f)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        smax = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i] == "Active"})
        power = [float(r[4]) for r in rows if r[4].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(power) if power else None}


def max_over_ranks(value: float, world: int, dev=None) -> float:
    """The largest value over all ranks (the slowest replica's time)."""
    t = torch.tensor([value], dtype=torch.float64)
    if world > 1:
        import torch.distributed as dist
        if dist.get_backend() == "nccl":
            t = t.to(dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def device_uuid(dev: torch.device):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


def workload_config(wl, world: int) -> dict:
    """The `config` object of a bench line: the workload alone, identical for
    the GPU arm and the reference arm on the same workload."""
    return {
        "workload": wl.name, "M": wl.M, "H": wl.H, "io_dtype": wl.dtype, "mode": wl.mode,
        "write_y": wl.write_y, "residual": wl.residual, "partials": wl.k,
        "weight_bias": wl.weight_bias,
        "parallelism": f"replicas{world}" if world > 1 else "single",
        "l2": (f"inputs larger than L2: each step moves {wl.algorithmic_bytes() / 1e6:.1f} MB; "
               "steps rotate over at least 8 input/output sets that together exceed 2x L2"
               if wl.algorithmic_bytes() > 128 * 2 ** 20 else
               "steps rotate over at least 8 input/output sets that together exceed 2x L2"),
    }


def kernel_name(kernel: int, cluster: int, vpt: int, form: int, wl) -> str:
    """Readable name of the kernel instance a launch shape runs (the shape
    as gnq_query_launch reports it)."""
    base = "row_kernel" if kernel == 1 else "stream_kernel"
    if wl.mode == "nvfp4":
        base += "_nvfp4"
    tname = {"bf16": "__nv_bfloat16", "fp16": "__half"}[wl.dtype]
    mode = {"none": "MODE_NONE", "fp8": "MODE_FP8", "nvfp4": "MODE_NVFP4",
            "mxfp8": "MODE_MXFP8"}[wl.mode]
    name = (f"gnq::{base}<{tname}, {mode}, parts={'true' if wl.k > 1 else 'false'}, VPT={vpt}, "
            f"{'packed' if form == 2 else 'fp32'}>")
    if kernel == 1 and cluster > 1:
        name += f" x {cluster}-CTA cluster"
    return name


def launched_kernel(gnq, wl) -> str:
    shape = gnq.query_launch(wl.M, wl.H, wl.mode, wl.dtype, k=wl.k, residual=wl.residual,
                             write_y=wl.write_y, weight_bias=wl.weight_bias)
    return kernel_name(*shape, wl)


# ----------------------------------------------------------------------------
# the GPU arm
# ----------------------------------------------------------------------------

def _device_inputs(wl, dev, exact: bool):
    """Inputs on the device: the seeded CPU recipe (exact), or the same
    distributions drawn with a seeded device generator (fast, for big shapes)."""
    if exact:
        return make_inputs(wl, dev)
    g = torch.Generator(device=dev).manual_seed(wl.seed)
    T = DTYPES[wl.dtype]
    M, H = wl.M, wl.H
    out = {}
    if wl.k > 1:
        out["x"] = (torch.randn(wl.k, M, H, generator=g, device=dev) * math.sqrt(wl.part_var)).to(T)
    else:
        out["x"] = (torch.randn(M, H, generator=g, device=dev) * math.sqrt(wl.x_var)).to(T)
    if wl.residual:
        r = torch.randn(M, H, generator=g, device=dev) * math.sqrt(wl.r_var)
        if wl.n_outliers:
            from nvfp4_quant_gemma_gb300.workloads import outlier_channels
            r[:, outlier_channels(wl).to(dev)] *= wl.outlier_mult
        out["residual"] = r.to(T)
    else:
        out["residual"] = None
    out["weight"] = (torch.randn(H, generator=g, device=dev) * math.sqrt(wl.w_var)).to(T)
    out["scale"] = torch.tensor([wl.scale], dtype=torch.float32, device=dev)
    out["eps"] = wl.eps
    return out


class Case:
    """Rotating input/output sets of one workload and the call that runs a step."""

    def __init__(self, gnq, wl, dev, exact_inputs: bool, l2_bytes: int):
        self.gnq, self.wl, self.dev = gnq, wl, dev
        base = _device_inputs(wl, dev, exact_inputs)
        self.w, self.scale, self.eps = base["weight"], base["scale"], base["eps"]
        per_set = wl.algorithmic_bytes()
        free = torch.cuda.mem_get_info(dev)[0]
        # At least eight sets: a set comes round again only after seven other
        # steps, by when no line of it is left in L2 -- not even those the
        # row kernel prefetches with the evict-last priority (with two sets
        # some were, and the large batches moved ~1 % fewer DRAM bytes).
        self.n_sets = max(8, min(64, math.ceil(2.5 * l2_bytes / per_set)))
        self.n_sets = max(1, min(self.n_sets, int(0.5 * free // max(1, 2 * per_set))))
        self.sets = []
        for i in range(self.n_sets):
            x = base["x"] if i == 0 else base["x"].clone()
            r = None if base["residual"] is None else (base["residual"] if i == 0 else base["residual"].clone())
            out = gnq.alloc_outputs(wl.M, wl.H, wl.mode, wl.write_y, x)
            self.sets.append((x, r, out))
        self.footprint = per_set * self.n_sets

    def step(self, i: int, stream=None):
        x, r, out = self.sets[i % self.n_sets]
        wl = self.wl
        if wl.weight_bias == 0.0:
            self.gnq.add_rms_norm_quant(x, r, self.w, self.eps, self.scale, wl.mode,
                                        write_y=wl.write_y, out=out, stream=stream)
        elif wl.k > 1:
            self.gnq.gemma_add_rms_norm_quant_parts(x, r, self.w, self.eps, self.scale, wl.mode,
                                                    write_y=wl.write_y, out=out, stream=stream)
        elif wl.mode == "none":
            self.gnq.gemma_add_rms_norm(x, r, self.w, self.eps, y=out[2], stream=stream)
        else:
            self.gnq.gemma_add_rms_norm_quant(x, r, self.w, self.eps, self.scale, wl.mode,
                                              write_y=wl.write_y, out=out, stream=stream)

    def graph(self, n: int, start: int = 0):
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(self.dev)
        s.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(s):
            self.step(0)  # first launch outside capture (library init)
        torch.cuda.current_stream(self.dev).wait_stream(s)
        torch.cuda.synchronize(self.dev)
        with torch.cuda.graph(g):
            for i in range(n):
                self.step(start + i)
        return g


def time_graph(g, dev, n_steps: int, barrier=None, soak_s: float = 0.0, sampler=None,
               profile_range: bool = False):
    """Replay g once inside CUDA events (after optional soak replays).  With
    profile_range the timed replay is also bracketed by cudaProfilerStart /
    Stop, so a profiler started with profiling off captures exactly it."""
    stream = torch.cuda.current_stream(dev)
    ctx = sampler if sampler is not None else _Null()
    with ctx:
        t_end = time.time() + soak_s
        while time.time() < t_end:
            g.replay()
            torch.cuda.synchronize(dev)
        if barrier:
            barrier()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        if profile_range:
            torch.cuda.profiler.start()
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        if profile_range:
            torch.cuda.profiler.stop()
        if barrier:
            barrier()
        ms = e0.elapsed_time(e1)
        t_end = time.time() + soak_s
        while time.time() < t_end:
            g.replay()
            torch.cuda.synchronize(dev)
    return ms


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        pass


def row_blocks(M: int, chunks: int) -> list[tuple[int, int]]:
    """Split M rows into at most `chunks` consecutive blocks whose starts are
    multiples of 128 rows (so an NVFP4 block-scale buffer splits at 128-row
    tile boundaries into contiguous pieces)."""
    per = -(-(-(-M // max(1, chunks))) // 128) * 128
    bounds, a = [], 0
    while a < M:
        bounds.append((a, min(M, a + per)))
        a += per
    return bounds


def e2e_measure(gnq, wl, dev, steps: int, warmup: int, barrier=None, graph: bool = True,
                chunks: int = 4, n_sets: int = 2, results: list | None = None, reps: int = 3,
                times: list | None = None):
    """Same metric through the public API with host buffers: every step copies
    its inputs from pinned host memory, runs the op, and reads its results
    back into pinned host memory.  A step's rows are cut into `chunks` row
    blocks (the op is row-wise); each block goes host -> device on a copy-in
    stream, through the op on a compute stream, and back on a copy-out
    stream, so the link carries both directions at once while the op runs on
    the blocks in between, across step boundaries too.  Device buffers and
    host result buffers rotate over `n_sets` sets; a block of a set is copied
    in again only after its previous results have been copied out.  With
    `graph` the steps are captured once into a CUDA graph and replayed (as a
    serving loop would), which removes the per-call host overhead but none of
    the transfers; otherwise they are issued eagerly.  The `steps` are timed
    `reps` times (the host link is shared with the machine's other work) and
    the median is returned; `times`, if given, receives every run's ms.
    `results`, if given, receives each set's host results ((q, block_scale,
    y), residual) after the timed steps, for checking."""
    inp = make_inputs(wl)
    n_host = 4
    host_in = []
    for i in range(n_host):
        x = inp["x"].clone().pin_memory()
        r = None if inp["residual"] is None else inp["residual"].clone().pin_memory()
        host_in.append((x, r))
    w = inp["weight"].to(dev)
    s = inp["scale"].to(dev)
    row_dim = 1 if wl.k > 1 else 0  # x_parts is (k, M, H)
    sets = []
    for _ in range(n_sets):
        xd = torch.empty_like(inp["x"], device=dev)
        rd = None if inp["residual"] is None else torch.empty_like(inp["residual"], device=dev)
        out = gnq.alloc_outputs(wl.M, wl.H, wl.mode, wl.write_y, xd)
        host_out = [None if t is None else torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                    for t in out]
        host_r = None if rd is None else torch.empty(rd.shape, dtype=rd.dtype, pin_memory=True)
        sets.append((xd, rd, out, host_out, host_r))
    h2d = sum(t.numel() * t.element_size() for t in host_in[0] if t is not None)
    d2h = sum(t.numel() * t.element_size() for t in sets[0][3] if t is not None)
    d2h += 0 if sets[0][4] is None else sets[0][4].numel() * sets[0][4].element_size()
    # k partials: one block (a row slice of (k, M, H) is not one contiguous tensor)
    bounds = row_blocks(wl.M, chunks if wl.k == 1 else 1)
    s_in, s_op, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    free = {}  # (set, block) -> event after that block's results were copied out

    def rows(t, a, e, dim=0):
        return t.narrow(dim, a, e - a)

    def one(i):
        b = i % n_sets
        hx, hr = host_in[i % n_host]
        xd, rd, out, host_out, host_r = sets[b]
        for j, (a, e) in enumerate(bounds):
            if (b, j) in free:
                s_in.wait_event(free[(b, j)])
            with torch.cuda.stream(s_in):
                rows(xd, a, e, row_dim).copy_(rows(hx, a, e, row_dim), non_blocking=True)
                if rd is not None:
                    rows(rd, a, e).copy_(rows(hr, a, e), non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(s_in)
            s_op.wait_event(ev)
            q, bs, y = out
            # the block's outputs: NVFP4 scales in whole 128-row tiles
            bs_e = bs.shape[0] if (bs is not None and wl.mode == "nvfp4" and e == wl.M) else e
            o = (None if q is None else rows(q, a, e),
                 None if bs is None or wl.mode == "fp8" else rows(bs, a, bs_e),
                 None if y is None else rows(y, a, e))
            xs, rs = rows(xd, a, e, row_dim), None if rd is None else rows(rd, a, e)
            with torch.cuda.stream(s_op):
                if wl.k > 1:
                    gnq.gemma_add_rms_norm_quant_parts(xs, rs, w, wl.eps, s, wl.mode,
                                                       write_y=wl.write_y, out=o)
                else:
                    gnq.gemma_add_rms_norm_quant(xs, rs, w, wl.eps, s, wl.mode,
                                                 write_y=wl.write_y, out=o)
            ev = torch.cuda.Event()
            ev.record(s_op)
            s_out.wait_event(ev)
            with torch.cuda.stream(s_out):
                for h, d in zip(host_out, o):
                    if d is not None:
                        hs = rows(h, a, bs_e) if d is o[1] else rows(h, a, e)
                        hs.copy_(d, non_blocking=True)
                if rd is not None:
                    rows(host_r, a, e).copy_(rs, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(s_out)
            free[(b, j)] = ev

    def run_steps(origin, n):
        # every stream starts after `origin`; `origin` then waits for all
        free.clear()
        for st in (s_in, s_op, s_out):
            st.wait_stream(origin)
        for i in range(n):
            one(i)
        for st in (s_in, s_op, s_out):
            origin.wait_stream(st)

    main = torch.cuda.current_stream(dev)
    run_steps(main, warmup)
    torch.cuda.synchronize(dev)
    g = None
    if graph:
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(main)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            run_steps(cap, steps)
        main.wait_stream(cap)
        g.replay()  # warm replay
        torch.cuda.synchronize(dev)
    runs = []
    for _ in range(max(1, reps)):
        if barrier:
            barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(main)
        if g is not None:
            g.replay()
        else:
            run_steps(main, steps)
        e1.record(main)
        torch.cuda.synchronize(dev)
        runs.append(e0.elapsed_time(e1))
    if times is not None:
        times.extend(runs)
    if results is not None:
        results.extend((st[3], st[4]) for st in sets)
    return statistics.median(runs), h2d, d2h


def e2e_zero_copy(gnq, wl, dev, steps: int, warmup: int, l2_bytes: int, barrier=None,
                  reps: int = 3):
    """Same metric with every buffer in pinned host memory: each step's
    kernel reads its inputs and writes its results through the host link
    (NVLink-C2C on a Grace-Blackwell node) with no separate copy.  Enough host
    sets rotate that their total is over 2.5x L2, so no step finds its inputs
    cached; the steps are captured in a CUDA graph and replayed, `reps` times
    (the median is returned)."""
    inp = make_inputs(wl)
    per_set = wl.algorithmic_bytes()
    n_sets = max(2, min(64, math.ceil(2.5 * l2_bytes / per_set)))
    w = inp["weight"].clone().pin_memory()
    sc = inp["scale"].clone().pin_memory()
    sets = []
    for _ in range(n_sets):
        x = inp["x"].clone().pin_memory()
        r = None if inp["residual"] is None else inp["residual"].clone().pin_memory()
        sets.append((x, r, gnq.alloc_outputs(wl.M, wl.H, wl.mode, wl.write_y, x)))
    x0, r0, out0 = sets[0]
    h2d = x0.numel() * x0.element_size() + (0 if r0 is None else r0.numel() * r0.element_size())
    d2h = sum(t.numel() * t.element_size() for t in out0 if t is not None)
    d2h += 0 if r0 is None else r0.numel() * r0.element_size()

    def one(i, st):
        x, r, out = sets[i % n_sets]
        if wl.k > 1:
            gnq.gemma_add_rms_norm_quant_parts(x, r, w, wl.eps, sc, wl.mode, write_y=wl.write_y,
                                               out=out, stream=st)
        else:
            gnq.gemma_add_rms_norm_quant(x, r, w, wl.eps, sc, wl.mode, write_y=wl.write_y,
                                         out=out, stream=st)

    main = torch.cuda.current_stream(dev)
    for i in range(warmup):
        one(i, main)
    torch.cuda.synchronize(dev)
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(main)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        for i in range(steps):
            one(i, cap)
    main.wait_stream(cap)
    g.replay()
    torch.cuda.synchronize(dev)
    runs = []
    for _ in range(max(1, reps)):
        if barrier:
            barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(main)
        g.replay()
        e1.record(main)
        torch.cuda.synchronize(dev)
        runs.append(e0.elapsed_time(e1))
    return statistics.median(runs), h2d, d2h


def host_link(dev, nbytes: int = 1 << 30, reps: int = 5, mix: tuple[int, int] | None = None) -> dict:
    """Copy-engine bandwidth between pinned host memory and the device:
    host->device, device->host, and both directions at once on two streams
    (best of `reps` copies of `nbytes`, CUDA events).  `mix` = (bytes in,
    bytes out): also one copy of each size at once, the two directions of a
    step's transfers alone (`step_mix_GB_s`, their total over the time)."""
    h_in = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h_out = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d_a = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_b = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def best(fn):
        t = []
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            main = torch.cuda.current_stream(dev)
            e0.record(main)
            fn(main)
            e1.record(main)
            torch.cuda.synchronize(dev)
            t.append(e0.elapsed_time(e1))
        return min(t)

    def h2d(main):
        d_a.copy_(h_in, non_blocking=True)

    def d2h(main):
        h_out.copy_(d_b, non_blocking=True)

    def both(main):
        for st in (s1, s2):
            st.wait_stream(main)
        with torch.cuda.stream(s1):
            d_a.copy_(h_in, non_blocking=True)
        with torch.cuda.stream(s2):
            h_out.copy_(d_b, non_blocking=True)
        main.wait_stream(s1)
        main.wait_stream(s2)

    gbs = lambda ms, n: n / (ms / 1e3) / 1e9
    out = {"h2d_GB_s": round(gbs(best(h2d), nbytes), 1),
           "d2h_GB_s": round(gbs(best(d2h), nbytes), 1),
           "bidirectional_GB_s": round(gbs(best(both), 2 * nbytes), 1),
           "how": f"cudaMemcpyAsync of {nbytes >> 20} MiB between pinned host memory and the "
                  f"device, best of {reps}; bidirectional: one copy each way on two streams"}
    del h_in, h_out, d_a, d_b
    if mix is not None:
        n_in, n_out = mix
        h_in = torch.empty(n_in, dtype=torch.uint8, pin_memory=True)
        h_out = torch.empty(n_out, dtype=torch.uint8, pin_memory=True)
        d_a = torch.empty(n_in, dtype=torch.uint8, device=dev)
        d_b = torch.empty(n_out, dtype=torch.uint8, device=dev)
        out["step_mix_GB_s"] = round(gbs(best(both), n_in + n_out), 1)
        out["how"] += (f"; step_mix: {n_in} bytes in and {n_out} bytes out at once, the copies "
                       "of one step without the op")
        del h_in, h_out, d_a, d_b
    return out


def link_ceiling(bytes_step: int, h2d: int, d2h: int, link: dict) -> float:
    """The end-to-end value the host link alone allows: a step's copies in
    and out overlapped at the measured one-way and two-way rates, and, where
    measured, at the rate of the step's own two copies running at once
    (each direction is slower while the other runs, so an uneven mix cannot
    use the whole two-way rate)."""
    t_one = max(h2d / (link["h2d_GB_s"] * 1e9), d2h / (link["d2h_GB_s"] * 1e9))
    t_two = (h2d + d2h) / (link["bidirectional_GB_s"] * 1e9)
    t_mix = (h2d + d2h) / (link["step_mix_GB_s"] * 1e9) if "step_mix_GB_s" in link else 0.0
    return bytes_step / max(t_one, t_two, t_mix) / 1e9


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or "unknown"."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith(("model name", "cpu part")):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_baseline(wl, budget_s: float = 10.0):
    """The oracle as it stands, on the host cores, over repeated passes of a
    row sample of the workload: about budget_s seconds with OpenMP over rows
    on every core, then about budget_s / 4 on one thread."""
    import numpy as np

    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    rows = min(wl.M, 256)
    sample = wl.with_rows(rows)
    inp = make_inputs(sample)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    x = bits(inp["x"])
    r = None if inp["residual"] is None else bits(inp["residual"])
    w = bits(inp["weight"])
    mode = {"fp8": oracle.MODE_FP8, "nvfp4": oracle.MODE_NVFP4, "mxfp8": oracle.MODE_MXFP8,
            "none": oracle.MODE_NONE}[wl.mode]
    dc = 0 if wl.dtype == "bf16" else 1

    def timed(n_threads, budget):
        oracle.set_threads(n_threads)
        passes = 0
        t0 = time.perf_counter()
        while True:
            oracle.gemma_add_rms_norm_quant(x, r, w, wl.eps, wl.scale, mode, dc,
                                            write_y=wl.write_y, weight_bias=wl.weight_bias)
            passes += 1
            el = time.perf_counter() - t0
            if el >= budget:
                return passes, el

    passes, el = timed(threads, budget_s)
    passes1, el1 = timed(1, budget_s / 4)
    oracle.set_threads(threads)
    per_pass = sample.algorithmic_bytes() / 1e9
    return {"value": per_pass * passes / el, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{passes} passes over {rows} rows of {wl.name} ({el:.1f} s)",
            "tokens_per_s": rows * passes / el,
            "single_thread_value": per_pass * passes1 / el1,
            "single_thread_sample": f"{passes1} passes ({el1:.1f} s, 1 thread)",
            "cpu_model": cpu_model()}


def run_gnq(args, rank: int, world: int, barrier):
    import nvfp4_quant_gemma_gb300 as gnq
    from nvfp4_quant_gemma_gb300 import build as libbuild

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    if libbuild.is_stale():
        libbuild.build()
    gnq.load()
    pol = [int(v) for v in args.policy.split(",")]
    gnq.set_launch_policy(*(pol + [0] * (4 - len(pol))))
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20
    peak, peak_kind = measured_peak()

    wl = all_workloads()[args.workload]
    case = Case(gnq, wl, dev, exact_inputs=True, l2_bytes=l2)
    g_warm = case.graph(max(args.warmup, 1))
    g_timed = case.graph(args.steps, start=args.warmup)
    g_warm.replay()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(device_uuid(dev)) if rank == 0 else None
    ms = time_graph(g_timed, dev, args.steps, barrier=barrier, soak_s=args.soak, sampler=sampler,
                    profile_range=True)
    ms_max = max_over_ranks(ms, world, dev)
    bytes_step = wl.algorithmic_bytes()
    value = bytes_step * args.steps * world / (ms_max / 1e3) / 1e9
    per_launch_s = ms / 1e3 / args.steps
    achieved = bytes_step / per_launch_s / 1e9
    n_sets, footprint = case.n_sets, case.footprint
    kernel = launched_kernel(gnq, wl) if args.policy == "0,0,0,0" else f"forced {args.policy}"

    e2e = None
    if not args.no_e2e:
        # end to end through the public API with host buffers
        del case, g_warm, g_timed
        torch.cuda.empty_cache()
        e2e_steps = max(1, min(args.steps, 500, int(16e9 // bytes_step)))
        chunks = 4
        zc_ms, h2d, d2h = e2e_zero_copy(gnq, wl, dev, e2e_steps, 3, l2, barrier)
        cp_runs = []
        cp_ms, _, _ = e2e_measure(gnq, wl, dev, e2e_steps, 3, barrier, graph=True, chunks=chunks,
                                  times=cp_runs)
        eager_ms, _, _ = e2e_measure(gnq, wl, dev, e2e_steps, 3, barrier, graph=False,
                                     chunks=chunks)
        gbs = lambda t: bytes_step * e2e_steps * world / (max_over_ranks(t, world, dev) / 1e3) / 1e9
        link = host_link(dev, mix=(h2d, d2h))
        vals = {"direct": gbs(zc_ms), "copy_engine": gbs(cp_ms), "eager": gbs(eager_ms)}
        e2e = {"value": round(vals["copy_engine"], 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": e2e_steps, "row_blocks": chunks,
               "runs_ms": [round(t, 3) for t in cp_runs],
               "direct_value": round(vals["direct"], 2),
               "eager_value": round(vals["eager"], 2),
               "host_link": link,
               "link_ceiling_value": round(link_ceiling(bytes_step, h2d, d2h, link) * world, 2),
               "how": "every step's inputs come from pinned host memory and its results go back "
                      "to pinned host memory, through the Python API. value: each step's rows in "
                      f"{chunks} blocks, every block copied in on one stream, run through the op "
                      "on a second and copied back on a third, so copies in, the op and copies "
                      "out overlap across blocks and steps; the steps replayed from a CUDA graph, "
                      "median of three timed runs (runs_ms). eager_value: the same issued from "
                      "Python call by call. direct_value: the kernels read and write the host "
                      "buffers over the host link themselves (no separate copy), graph-replayed. "
                      "link_ceiling_value: the value the measured copy-engine rates of the host "
                      "link allow for this step's bytes in and out (host_link.step_mix_GB_s: "
                      "the step's two copies alone, at once)."}

    if rank != 0:
        return None
    # the recorded traffic is the automatic launch's; a forced shape has none
    traffic = recorded_traffic(wl.name) if args.policy == "0,0,0,0" else None
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded normals; no dataset or weights involved)",
        "config": workload_config(wl, world),
        "tokens_per_s": wl.M * args.steps * world / (ms_max / 1e3),
        "us_per_call": ms_max / args.steps * 1e3,
        "pct_of_peak": round(100 * achieved / peak, 1),
        "pct_of_nominal_8TBs": round(100 * achieved / 8000.0, 1),
        "timing": (f"K launches captured in one CUDA graph over {n_sets} rotating input/output "
                   f"sets ({footprint / 1e6:.0f} MB > 2x L2 of {l2 / 1e6:.0f} MB), CUDA events on "
                   "the capture stream"),
        "roofline": {
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "peak_kind": peak_kind,
            "algorithmic_bytes_per_launch": bytes_step,
            "kernel": kernel,
            "traffic_source": "profiles/dram_traffic.txt (ncu, steady state)" if traffic else None,
        },
        "gpu_launches": args.steps,
    }
    if e2e is not None:
        line["e2e"] = e2e
    line["clocks"] = sampler.summary() if sampler else None
    if world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_budget)
    if world == 1 and not args.no_table:
        line["workloads"] = workload_table(gnq, dev, l2, peak)
    if world == 1 and not args.no_sweep:
        line["small_m_sweep"] = small_m_sweep(gnq, dev, l2, peak)
        line["pdl_consumer_sweep"] = pdl_consumer_sweep(gnq, dev, l2)
        line["dependent_launch_floor"] = dependent_launch_floor(gnq, dev)
    return line


def time_case(case, dev) -> tuple[float, int]:
    """Microseconds per call of a workload case: a CUDA graph of n back-to-back
    launches over its rotating sets, n sized for ~0.3 ms of work."""
    probe = case.graph(max(2, case.n_sets))
    probe.replay()
    torch.cuda.synchronize(dev)
    t = time_graph(probe, dev, case.n_sets) / case.n_sets
    n = int(min(4000, max(20, 0.3e3 / max(t, 1e-4))))
    g = case.graph(n)
    g.replay()
    torch.cuda.synchronize(dev)
    ms = time_graph(g, dev, n)
    del probe, g
    return ms / n * 1e3, n


def workload_table(gnq, dev, l2, peak):
    """Every workload: the five configurations and the further variants
    (MXFP8, plain RMSNorm, norm only) at their shapes."""
    rows = []
    for name, wl in all_workloads().items():
        case = Case(gnq, wl, dev, exact_inputs=(wl.M * wl.H <= 2 ** 22), l2_bytes=l2)
        us, n = time_case(case, dev)
        b = wl.algorithmic_bytes()
        gbs = b / (us / 1e6) / 1e9
        rows.append({"workload": name, "kind": "config" if name in WORKLOADS else "variant",
                     "kernel": launched_kernel(gnq, wl),
                     "us_per_call": round(us, 3), "GB_s": round(gbs, 1),
                     "frac_of_peak": round(gbs / peak, 4), "tokens_per_s": round(wl.M / (us / 1e6)),
                     "bytes_per_call": b, "launches_timed": n, "sets": case.n_sets,
                     "dram_traffic_per_launch": recorded_traffic(name)})
        del case
        torch.cuda.empty_cache()
    return rows


# launch shapes compared by the small-batch sweep: (label, kernel, cluster); for
# the streaming kernel `cluster` is the least number of rows per CTA
SWEEP_SHAPES = (("auto", 0, 0), ("row_cluster2", 1, 2), ("row_cluster4", 1, 4), ("stream", 2, 0),
                ("stream_2rows", 2, 2))


def small_m_sweep(gnq, dev, l2, peak, modes=("fp8", "nvfp4"), m_values=SMALL_M):
    """Latency for M = 1 .. 8192 rows at H = 5120 (bf16, residual, y), in the
    static-FP8 and the NVFP4 mode: the automatic launch shape against
    split-row clusters of 2 and 4 CTAs (partial sums of squares exchanged
    through distributed shared memory), the persistent streaming grid, and
    that grid with at least two rows per CTA (the second row's copy in
    flight while the first is computed)."""
    rows = []
    try:
        for mode in modes:
            for M in m_values:
                wl = sweep_workload(mode, M)
                case = Case(gnq, wl, dev, exact_inputs=(M * wl.H <= 2 ** 24), l2_bytes=l2)
                row = {"mode": mode, "M": M, "H": wl.H}
                shape = gnq.query_launch(M, wl.H, wl.mode, wl.dtype, residual=wl.residual,
                                         write_y=wl.write_y)
                row["auto_shape"] = kernel_name(*shape, wl)
                for label, kernel, cluster in SWEEP_SHAPES:
                    gnq.set_launch_policy(kernel, cluster, 0, 0)
                    us, _ = time_case(case, dev)
                    row[label + "_us"] = round(us, 3)
                gnq.set_launch_policy(0, 0, 0, 0)
                row["auto_GB_s"] = round(wl.algorithmic_bytes() / (row["auto_us"] / 1e6) / 1e9, 1)
                rows.append(row)
                del case
                torch.cuda.empty_cache()
    finally:
        gnq.set_launch_policy(0, 0, 0, 0)
    return rows


# launches compared with a consumer: (label, programmatic dependent launch on)
PDL_POLICIES = (("pdl_trigger_early", True), ("no_pdl", False))
PDL_M = (1, 16, 64, 128, 152, 192, 256, 512, 2048, 8192)
CONSUMER_WEIGHT_PER_CTA = 32768  # bytes each consumer CTA reads before its wait


def time_pairs(case, dev, consumer, probe_n: int = 8) -> float:
    """Microseconds per (call, consumer) pair: a CUDA graph of n pairs, each
    call followed by the stand-in consumer of its codes."""
    def graph(n):
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):
            case.step(0)
            consumer(0)
        torch.cuda.current_stream(dev).wait_stream(s)
        torch.cuda.synchronize(dev)
        with torch.cuda.graph(g):
            for i in range(n):
                case.step(i)
                consumer(i)
        g.replay()
        torch.cuda.synchronize(dev)
        return g
    g = graph(probe_n)
    t = time_graph(g, dev, probe_n) / probe_n
    n = int(min(2000, max(20, 0.3e3 / max(t, 1e-4))))
    g = graph(n)
    return time_graph(g, dev, n) / n * 1e3


def pdl_consumer_sweep(gnq, dev, l2, modes=("fp8", "nvfp4"), m_values=PDL_M):
    """Programmatic dependent launch with a real consumer: each call (H =
    5120, bf16, residual, y) is followed by a stand-in for the next layer's
    first kernel (one CTA per SM, launched as a programmatic dependent; it
    reads 32 KB of its own weight per CTA before it waits, then the call's
    codes), with the calls launched as programmatic dependents that let the
    consumer launch right after their own wait, and as plain launches."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    wt = torch.randint(0, 255, (sms * CONSUMER_WEIGHT_PER_CTA,), dtype=torch.uint8, device=dev)
    out = torch.empty(sms * 256, dtype=torch.int32, device=dev)
    rows = []
    try:
        for mode in modes:
            for M in m_values:
                wl = sweep_workload(mode, M)
                case = Case(gnq, wl, dev, exact_inputs=(M * wl.H <= 2 ** 24), l2_bytes=l2)

                def consumer(i, case=case):
                    q = case.sets[i % case.n_sets][2][0]
                    gnq.pdl_consumer(q, wt, out, sms)

                row = {"mode": mode, "M": M, "H": wl.H}
                for label, pol in PDL_POLICIES:
                    gnq.set_pdl(pol)
                    row[label + "_us"] = round(time_pairs(case, dev, consumer), 3)
                gnq.set_pdl(True)
                rows.append(row)
                del case
                torch.cuda.empty_cache()
    finally:
        gnq.set_pdl(True)
    return rows


def dependent_launch_floor(gnq, dev, n: int = 2000) -> dict:
    """Time per kernel of a chain of n programmatic dependents that move
    almost nothing (the stand-in consumer, one CTA, reading 16 bytes after
    its wait): the launch-and-dependency cost any dependent call pays on
    this GPU before it moves data."""
    q = torch.zeros(16, dtype=torch.uint8, device=dev)
    no_weight = torch.empty(0, dtype=torch.uint8, device=dev)
    out = torch.empty(256, dtype=torch.int32, device=dev)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        gnq.pdl_consumer(q, no_weight, out, 1)
    torch.cuda.current_stream(dev).wait_stream(s)
    torch.cuda.synchronize(dev)
    with torch.cuda.graph(g):
        for _ in range(n):
            gnq.pdl_consumer(q, no_weight, out, 1)
    g.replay()
    torch.cuda.synchronize(dev)
    return {"us_per_kernel": round(time_graph(g, dev, n) / n * 1e3, 3), "kernels": n,
            "how": "a CUDA graph of dependent launches of the stand-in consumer (one CTA, "
                   "16 bytes read after its wait, nothing before it), CUDA events"}


# ----------------------------------------------------------------------------
# the reference arm: the CPU oracle
# ----------------------------------------------------------------------------

def run_reference(args, rank: int):
    if rank != 0:
        return None
    import numpy as np

    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    oracle.set_threads(threads)
    wl = all_workloads()[args.workload]
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    mode = {"fp8": oracle.MODE_FP8, "nvfp4": oracle.MODE_NVFP4, "mxfp8": oracle.MODE_MXFP8,
            "none": oracle.MODE_NONE}[wl.mode]
    dc = 0 if wl.dtype == "bf16" else 1
    # size one step so the K steps take about args.ref_budget seconds
    probe = wl.with_rows(min(wl.M, 16))
    pin = make_inputs(probe)
    t0 = time.perf_counter()
    oracle.gemma_add_rms_norm_quant(bits(pin["x"]), None if pin["residual"] is None else bits(pin["residual"]),
                                    bits(pin["weight"]), wl.eps, wl.scale, mode, dc, write_y=wl.write_y,
                                    weight_bias=wl.weight_bias)
    per_row = (time.perf_counter() - t0) / probe.M
    rows = int(max(1, min(wl.M, args.ref_budget / max(1, args.steps) / max(per_row, 1e-9))))
    sample = wl.with_rows(rows)
    inp = make_inputs(sample)
    x = bits(inp["x"])
    r = None if inp["residual"] is None else bits(inp["residual"])
    w = bits(inp["weight"])
    for _ in range(args.warmup):
        oracle.gemma_add_rms_norm_quant(x, r, w, wl.eps, wl.scale, mode, dc, write_y=wl.write_y,
                                        weight_bias=wl.weight_bias)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.gemma_add_rms_norm_quant(x, r, w, wl.eps, wl.scale, mode, dc, write_y=wl.write_y,
                                        weight_bias=wl.weight_bias)
    el = time.perf_counter() - t0
    value = sample.algorithmic_bytes() * args.steps / el / 1e9
    sample_txt = f"{rows} of {wl.M} rows of {wl.name} per step"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded normals)",
        "config": workload_config(wl, int(os.environ.get("WORLD_SIZE", "1"))),
        "sample": sample_txt,
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample_txt, "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


# ----------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gnq", choices=["gnq", "reference"])
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(all_workloads()))
    ap.add_argument("--soak", type=float, default=0.6,
                    help="seconds of identical replays before and after the timed replay, "
                         "so the clock sampler sees the load")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--ref-budget", type=float, default=40.0)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-table", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the small-batch latency sweep")
    ap.add_argument("--policy", default="0,0,0,0",
                    help="forced launch shape kernel,cluster,vpt,form (0 = automatic)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        # the CPU oracle: rank 0 alone runs it; other ranks exit without work
        line = run_reference(args, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    barrier = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group(backend)
        barrier = dist.barrier

    line = run_gnq(args, rank, world, barrier)
    if line is not None and rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
