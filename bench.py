"""Benchmark: NVFP4 quantize throughput (GB/s of BF16-in ideal bytes) on GB300.

One step = the whole hot path on one batch of seeded synthetic input resident in HBM: every
kernel a caller runs to turn a BF16 tensor into NVFP4 codes, E4M3 scales and FP32 global
scales. Grouped (MoE) workloads, the default: the per-expert amax pass (nvfp4_amax_grouped)
then the grouped quantize kernel with those maxima (nvfp4_quantize_grouped), the two launches
nvfp4_quantize_grouped makes on its own. Plain tensors: by default one nvfp4_quantize launch
that computes the amax itself (fused_amax), or with --pipeline two_pass the amax kernel
(nvfp4_amax) followed by the quantize kernel.
Ideal bytes per step = one BF16 read + code writes + scale writes (the metric's roofline
bytes). Between timed steps L2 holds none of the step's data: by default (--l2 rotate) the steps
cycle through K input/output sets whose total is at least three times the L2 size (inputs
larger than L2), with --l2 flush a 256 MiB buffer is written before every step. Device time
comes from CUDA events on the launching stream: one pair around the K back-to-back steps (with
the flush, a pair around every step). Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--pipeline fused|two_pass] [--l2 rotate|flush]
"""
import argparse
import dataclasses
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from nvfp4_block_scaled_quantize_gb300 import workloads  # noqa: E402

# the largest configuration, and the pages' headline workload kind (grouped MoE row + col
# RHT/SR quantization); the others through --workload
DEFAULT_WORKLOAD = "moe_64experts_32768x7168_row_rtne_col_rht_sr"
METRIC = "NVFP4 quantize GB/s (BF16 in) and fraction of GB300 HBM roofline, 1 GPU"
FLUSH_BYTES = 256 << 20


def ideal_bytes(w: workloads.Workload, rows=None, offsets=None) -> int:
    """One BF16 read + codes (half a byte per element) + scales (1/16 byte per element) per
    produced orientation. Grouped columnwise outputs count their padded tokens."""
    M = w.rows if rows is None else rows
    N = w.cols
    b = 2 * M * N
    if w.rowwise:
        b += M * N // 2 + M * N // 16
    if w.columnwise:
        P = M
        if w.grouped and offsets is not None:
            P = int(sum((int(c) + 15) // 16 * 16 for c in np.diff(np.concatenate([[0], offsets]))))
        b += P * N // 2 + P * N // 16
    return b


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


KERNEL_SOURCES = ("quantize_kernel.cuh", "fused_amax.cuh", "nvfp4_device.cuh", "nvfp4_internal.h")


def _code_only(text: str) -> str:
    """C++ source without comments and whitespace (string literals in these files hold no
    comment markers), so that only code changes change the digest."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return re.sub(r"\s+", "", text)


def kernel_source_digest() -> str:
    """sha256 (first 16 hex digits) over the tile kernel's sources, code only, in a fixed order."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "nvfp4_block_scaled_quantize_gb300", "csrc", name)) as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def kernel_traffic(workload: str, pipeline: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel, workload and
    pipeline, valid only while the kernel sources are unchanged (the summary records their
    digest)."""
    summary = os.path.join(ROOT, "profiles", "quantize_tiles_%s_%s.txt" % (workload, pipeline))
    if not os.path.exists(summary):
        return None
    fields = {}
    for line in open(summary):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    if fields.get("source_sha256_16", "").split()[:1] != [kernel_source_digest()]:
        return None
    try:
        return int(fields["dram_bytes_per_launch"].split()[0])
    except (KeyError, ValueError, IndexError):
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons; summary() keeps the samples that
    arrived between mark_start() and mark_end() (the timed region)."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.lines = []
        self.window = (0.0, float("inf"))

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def mark_start(self):
        self.window = (time.monotonic(), float("inf"))

    def mark_end(self):
        self.window = (self.window[0], time.monotonic())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, ln in self.lines:
            if not self.window[0] <= t <= self.window[1]:
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value):
    if world == 1:
        return value
    import torch.distributed as dist
    dev = torch.device("cuda") if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(ideal_bytes_per_step, steps, world, total_s):
    """Whole-job throughput: every rank's bytes (replicas: the same work per rank) over the
    slowest rank's timed region."""
    return ideal_bytes_per_step * steps * world / total_s / 1e9


def quant_kwargs(w, inp):
    return dict(rowwise=w.rowwise, columnwise=w.columnwise, block2d=w.block2d,
                rht_col=w.rht_col, sign_mask=inp["sign_mask"], seed=inp["seed"],
                round_row="sr" if w.round_row_sr else "rn",
                round_col="sr" if w.round_col_sr else "rn")


def _oracle_run(w, inp, rows):
    """The oracle, as it stands, on the first `rows` rows of the workload (amax + outputs)."""
    import oracle
    xb = oracle.as_bf16_bits(inp["x"])[:rows]
    t0 = time.perf_counter()
    if w.grouped:
        off = np.minimum(inp["offsets"], rows).astype(np.int32)
        oracle.quantize_grouped(xb, off, rowwise=w.rowwise, columnwise=w.columnwise,
                                round_row_sr=w.round_row_sr, round_col_sr=w.round_col_sr,
                                rht_col=w.rht_col, sign_mask=inp["sign_mask"], seed=inp["seed"],
                                block2d=w.block2d)
    else:
        oracle.quantize(xb, oracle.Config(rowwise=w.rowwise, columnwise=w.columnwise,
                                          block2d=w.block2d, round_row_sr=w.round_row_sr,
                                          round_col_sr=w.round_col_sr, rht_col=w.rht_col,
                                          sign_mask=inp["sign_mask"], seed=inp["seed"]))
    return time.perf_counter() - t0


def cpu_model() -> str:
    """The host CPU's model name (lscpu's, else /proc/cpuinfo's, else the platform's)."""
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_run_threads(w, inp, rows, threads):
    """The oracle's own functions on `threads` host threads over 64-row chunks of the first
    `rows` rows: the amax per chunk, then every chunk quantized with the tensor's amax (ctypes
    releases the GIL during each call). Plain tensors only. RTNE outputs equal the one-thread
    run's; under SR each chunk's block indices restart at zero (same work, another stream)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    xb = oracle.as_bf16_bits(inp["x"])[:rows]
    step = max(64, -(-rows // threads) // 64 * 64)
    chunks = [xb[r:r + step] for r in range(0, rows, step)]
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as pool:
        amax = max(pool.map(oracle.amax, chunks))
        amax_c = (max(pool.map(lambda c: oracle.amax_rht(c, inp["sign_mask"]), chunks))
                  if w.rht_col else amax)

        def one(c):
            if w.block2d:
                return oracle.quantize_2d(c, amax_value=amax)
            if w.rowwise:
                oracle.quantize_rowwise(c, amax_value=amax, sr=w.round_row_sr, seed=inp["seed"])
            if w.columnwise:
                oracle.quantize_colwise(c, amax_value=amax_c, rht=w.rht_col,
                                        sign_mask=inp["sign_mask"], sr=w.round_col_sr,
                                        seed=inp["seed"])
        list(pool.map(one, chunks))
    return time.perf_counter() - t0


def cpu_sample_rows(w, inp, budget_s):
    """Rows (a multiple of 64) of the workload the oracle processes in about budget_s."""
    rows = 64
    dt = _oracle_run(w, inp, rows)
    while dt < budget_s / 8 and rows < w.rows:
        rows = min(w.rows, rows * 4)
        dt = _oracle_run(w, inp, rows)
    rows = int(min(w.rows, max(64, rows * budget_s / max(dt, 1e-6) // 64 * 64)))
    return rows


def cpu_baseline(w, inp, budget_s=15.0):
    """Oracle throughput on a bounded sample, in the metric's unit (ideal bytes / s): on every
    host core (threads over row chunks; grouped tensors on one), and on one core."""
    rows = cpu_sample_rows(w, inp, budget_s)
    dt1 = _oracle_run(w, inp, rows)
    off = np.minimum(inp["offsets"], rows) if w.grouped else None
    b = ideal_bytes(w, rows, off)
    cores = 1 if w.grouped else host_cores()
    dtn = dt1 if cores == 1 else _oracle_run_threads(w, inp, rows, cores)
    return {"value": b / dtn / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(), "single_core_value": b / dt1 / 1e9,
            "sample": "first %d of %d rows of %s (amax + every output): %.2f s on %d cores "
                      "(threads over 64-row chunks), %.2f s on 1 core"
                      % (rows, w.rows, w.name, dtn, cores, dt1)}


def run_reference(args, world, rank):
    """--impl reference: the oracle on the host cores, rank 0 only (the other ranks exit)."""
    if rank != 0:
        return
    w = workloads.WORKLOADS[args.workload]
    inp = workloads.make_input(w)
    cores = 1 if w.grouped else host_cores()
    # seconds per step: about 100 s of oracle work for the whole run (small samples scale
    # worse than linearly over the threads, so the run takes somewhat longer)
    budget = min(10.0, 100.0 / (args.steps + args.warmup))
    rows = cpu_sample_rows(w, inp, budget * cores)
    off = np.minimum(inp["offsets"], rows) if w.grouped else None
    b = ideal_bytes(w, rows, off)
    times = []
    for i in range(args.warmup + args.steps):
        dt = (_oracle_run(w, inp, rows) if cores == 1
              else _oracle_run_threads(w, inp, rows, cores))
        if i >= args.warmup:
            times.append(dt)
    value = b * len(times) / sum(times) / 1e9
    sample = "first %d of %d rows of %s per step (amax + every output), %d core%s%s" % (
        rows, w.rows, w.name, cores, "" if cores == 1 else "s",
        "" if cores == 1 else " (threads over 64-row chunks)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": statistics.mean(times) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "sample_rows": rows},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "cpu_model": cpu_model(), "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def nbytes(*tensors):
    return sum(t.numel() * t.element_size() for t in tensors)


def rotation_sets(set_bytes, l2_bytes):
    """The fewest input/output sets of set_bytes each that together hold 3 x l2_bytes."""
    return max(1, -(-3 * l2_bytes // set_bytes))


def l2_plan(args, dev, set_bytes):
    """How the timed steps keep their data out of L2. --l2 rotate (default): K input/output sets
    with K x set_bytes >= 3 x L2 and step j on set j % K, so a step's data was last touched three
    L2 capacities earlier (inputs larger than L2); --l2 flush: one set, and a 256 MiB buffer
    written before every step. Returns (K, the flush buffer or None, the note for the config)."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    if args.l2 == "flush":
        return (1, torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev),
                "flushed before every timed step (256 MiB write)")
    k = rotation_sets(set_bytes, l2)
    return k, None, ("inputs larger than L2: %d rotating input/output sets of %.0f MiB (%.1fx "
                     "the %.0f MiB L2), no flush" % (k, set_bytes / 2**20, k * set_bytes / l2,
                                                     l2 / 2**20))


def clear_l2(flush):
    if flush is not None:
        flush.zero_()


def workload_of(args):
    """The named workload, or with --rows a smaller case of it (same distribution and options;
    grouped inputs keep their expert count over fewer tokens), for profiling captures."""
    w = workloads.WORKLOADS[args.workload]
    return dataclasses.replace(w, rows=args.rows) if args.rows else w


def run_ours(args, world, rank, local):
    from nvfp4_block_scaled_quantize_gb300 import api, _lib
    _lib.load()
    dev = torch.device("cuda", local)
    w = workload_of(args)
    inp = workloads.make_input(w)
    x = inp["x"].to(dev)
    kw = quant_kwargs(w, inp)
    kw["fast_math"] = args.fast_math
    ideal = ideal_bytes(w, offsets=inp.get("offsets"))
    stream = torch.cuda.current_stream(dev)

    if w.grouped:
        offsets = torch.from_numpy(inp["offsets"]).to(dev)
        cap = int(sum((int(c) + 15) // 16 * 16 for c in np.diff(np.concatenate([[0], inp["offsets"]]))))
        alloc = lambda: api.alloc_outputs(w.rows, w.cols, dev, w.rowwise, w.columnwise,
                                          col_ld=cap, groups=w.experts)
    else:
        alloc = lambda: api.alloc_outputs(w.rows, w.cols, dev, w.rowwise, w.columnwise)
    out = alloc()
    n_sets, flush, l2_note = l2_plan(args, dev, nbytes(x, *out.values()))
    xs, outs = [x], [out]
    for _ in range(n_sets - 1):
        xs.append(x.clone())
        outs.append(alloc())

    if w.grouped:
        # the two launches of nvfp4_quantize_grouped, made through the public calls so that
        # events can sit between them: the per-expert amax pass, then the quantize kernel
        def step(j, ev=None):
            if ev:
                ev[0].record(stream)
            xj = xs[j % n_sets]
            a_row, a_col = api.nvfp4_amax_grouped(xj, offsets, rht_col=w.rht_col,
                                                  sign_mask=kw["sign_mask"])
            if ev:
                ev[1].record(stream)
            api.nvfp4_quantize_grouped(xj, offsets, col_capacity=cap, out=outs[j % n_sets],
                                       amax_row=a_row, amax_col=a_col, **kw)
            if ev:
                ev[2].record(stream)
        launches_per_step = 2
        kernel_split = True
    else:
        rht_amax = w.rht_col

        if args.pipeline == "fused":
            def step(j, ev=None):
                if ev:
                    ev[0].record(stream)  # one launch: the step and the kernel are the same span
                api.nvfp4_quantize(xs[j % n_sets], out=outs[j % n_sets], fused_amax=True, **kw)
                if ev:
                    ev[2].record(stream)
            launches_per_step = 1
        else:
            def step(j, ev=None):
                if ev:
                    ev[0].record(stream)
                xj = xs[j % n_sets]
                a_row, a_col = api.nvfp4_amax(xj, rht_col=rht_amax, sign_mask=kw["sign_mask"])
                if ev:
                    ev[1].record(stream)
                api.nvfp4_quantize(xj, amax_row=a_row, amax_col=a_col, out=outs[j % n_sets], **kw)
                if ev:
                    ev[2].record(stream)
            launches_per_step = 2
        kernel_split = True

    # With rotating sets the K timed steps run back to back between one pair of events (events
    # between launches would serialize them). A second pass with events around every step
    # gives the per-step spread and, for two passes, the quantize kernel alone; with the flush
    # the timed region itself uses per-step events, so that the flush writes stay outside.
    per_step_timed = args.l2 == "flush"
    n_ev = args.steps if per_step_timed else min(args.steps, 1000)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_ev)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index if dev.index is not None else 0) as clocks:
        time.sleep(0.3)  # the sampler is up before the GPU work starts
        clocks.mark_start()  # the record covers the warm-up and the timed region
        for j in range(args.warmup):
            clear_l2(flush)
            step(j)
        torch.cuda.synchronize(dev)
        status, bits = api.nvfp4_get_status(dev)
        if status != 0:
            raise RuntimeError("device status %d (bits %#x) after warm-up" % (status, bits))
        barrier(world)
        torch.cuda.synchronize(dev)
        if per_step_timed:
            for i in range(args.steps):
                clear_l2(flush)
                step(args.warmup + i, events[i])
        else:
            t_start.record(stream)
            for i in range(args.steps):
                step(args.warmup + i)
            t_end.record(stream)
        torch.cuda.synchronize(dev)
        clocks.mark_end()
        time.sleep(0.05)
    barrier(world)
    if not per_step_timed:
        for i in range(n_ev):
            step(args.warmup + args.steps + i, events[i])
        torch.cuda.synchronize(dev)
    status, bits = api.nvfp4_get_status(dev)
    if status != 0:
        raise RuntimeError("device status %d (bits %#x) after the timed steps" % (status, bits))
    step_ms = [e[0].elapsed_time(e[2]) for e in events]
    if kernel_split:
        quant_ms = ([e[0].elapsed_time(e[2]) for e in events]
                    if args.pipeline == "fused" and not w.grouped
                    else [e[1].elapsed_time(e[2]) for e in events])
    total_s = (sum(step_ms) if per_step_timed else t_start.elapsed_time(t_end)) / 1e3
    total_s = max_over_ranks(world, total_s)
    value = aggregate_gbs(ideal, args.steps, world, total_s)

    # end to end through the public API: pinned host input -> device -> quantize -> pinned host.
    # Plain tensors go through the host pipeline (the copy in of one step overlaps the copy out
    # of the previous one), grouped ones through its grouped form (the expert offsets copied in
    # with x).
    x_host = inp["x"].pin_memory()
    h2d = x_host.numel() * 2
    d2h = sum(v.numel() * v.element_size() for v in out.values())
    if w.grouped:
        offsets_host = torch.from_numpy(np.ascontiguousarray(inp["offsets"], dtype=np.int32))
        h2d += offsets_host.numel() * 4
        pipe = api.GroupedHostPipeline(w.rows, w.cols, w.experts, cap, depth=2, **kw)
        host_out = pipe.alloc_host_outputs()
        e2e_step = lambda: pipe.submit(x_host, offsets_host, host_out)  # noqa: E731
        e2e_join = pipe.join
    else:
        pipe = api.HostPipeline(w.rows, w.cols, depth=2, fused_amax=args.pipeline == "fused",
                                **kw)
        host_out = pipe.alloc_host_outputs()
        e2e_step = lambda: pipe.submit(x_host, host_out)  # noqa: E731
        e2e_join = pipe.join

    for _ in range(max(1, args.warmup)):
        e2e_step()
    e2e_join()
    torch.cuda.synchronize(dev)
    e2e_steps = min(args.steps, 200)   # each step moves ~100 MiB over the host link
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e2e_join()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_s = max_over_ranks(world, e0.elapsed_time(e1) / 1e3)
    e2e_value = ideal * e2e_steps * world / e2e_s / 1e9
    pipe.close()

    if rank != 0:
        return
    hbm, peak_kind = peaks()
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_s * 1e3 / args.steps,
        "elements_per_s": w.rows * w.cols * args.steps * world / total_s,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "shape": [w.rows, w.cols],
                   **({"rows_override": args.rows} if args.rows else {}),
                   "ideal_bytes_per_step": ideal,
                   "pipeline": ("one launch: amax phase, grid barrier, quantize phase"
                                if args.pipeline == "fused" and not w.grouped else
                                "per-expert amax pass + grouped quantize pass (two launches)"
                                if w.grouped else "amax pass + quantize pass (two launches)"),
                   "math": "fast (rcp.approx multipliers%s)" % (
                       ", FP32 RHT" if w.rht_col else "") if args.fast_math and not w.block2d
                           else "exact",
                   "l2": l2_note,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "gpu_launches": launches_per_step * args.steps,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "path": ("nvfp4_host_pipeline_*_grouped" if w.grouped else "nvfp4_host_pipeline")
                        + " depth 2 (copies of consecutive steps overlap)"},
        "clocks": clocks.summary(),
    }
    line["step_us"] = {"min": min(step_ms) * 1e3, "median": statistics.median(step_ms) * 1e3,
                       "max": max(step_ms) * 1e3,
                       "from": ("the timed steps" if per_step_timed else
                                "%d further steps with events around each (events between "
                                "launches serialize them)" % n_ev)}
    if kernel_split:
        # the single launch is the step, so its duration is the timed region's per-step time;
        # the two-pass pipeline's quantize kernel is timed alone by the events around it
        fused_step = args.pipeline == "fused" and not w.grouped
        qk = (total_s / args.steps if fused_step and not per_step_timed
              else statistics.mean(quant_ms) / 1e3)
        achieved = ideal / qk / 1e9
        line["roofline"] = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                            "frac": achieved / hbm, "peak_kind": peak_kind,
                            "kernel": "quantize_tiles_kernel",
                            "kernel_us": qk * 1e6,
                            "traffic": (None if args.fast_math
                                        else kernel_traffic(w.name, "fused" if fused_step
                                                            else "two_pass"))}
        if not fused_step:
            line["amax_pass_us"] = statistics.mean([e[0].elapsed_time(e[1]) for e in events]) * 1e3
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inp)
    print(json.dumps(line), flush=True)


MX_METRIC = "MX quantize GB/s (BF16 in) and fraction of GB300 HBM roofline, 1 GPU"


def mx_ideal_bytes(w, fmt, rows=None) -> int:
    """One BF16 read + codes (1 byte per element for FP8, half for FP4) + E8M0 scales (1/32
    byte per element) per produced orientation."""
    M = w.rows if rows is None else rows
    n = M * w.cols
    per = (n // 2 if fmt == "e2m1" else n) + n // 32
    return 2 * n + per * (int(w.rowwise) + int(w.columnwise))


def mx_cpu_baseline(w, inp, fmt, budget_s=15.0):
    """The oracle's MX functions on a bounded row sample, threads over 64-row chunks (blocks
    are independent: no amax)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    xb = oracle.as_bf16_bits(inp["x"])

    def run(rows, threads):
        chunks = [xb[r:r + 64] for r in range(0, rows, 64)]

        def one(c):
            if w.rowwise:
                oracle.mx_quantize_rowwise(c, fmt)
            if w.columnwise:
                oracle.mx_quantize_colwise(c, fmt)
        t0 = time.perf_counter()
        with ThreadPoolExecutor(max_workers=threads) as pool:
            list(pool.map(one, chunks))
        return time.perf_counter() - t0
    rows = 64
    dt = run(rows, 1)
    while dt < budget_s / 8 and rows < w.rows:
        rows = min(w.rows, rows * 4)
        dt = run(rows, 1)
    cores = host_cores()
    rows = int(min(w.rows, max(64, rows * budget_s * cores / max(dt, 1e-6) // 64 * 64)))
    dtn = run(rows, cores)
    b = mx_ideal_bytes(w, fmt, rows)
    return {"value": b / dtn / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": "first %d of %d rows of %s, MX %s (every output): %.2f s on %d cores "
                      "(threads over 64-row chunks)" % (rows, w.rows, w.name, fmt, dtn, cores)}


def run_mx(args, world, rank, local):
    """--mx FMT: the MX quantizer on the workload's shape and orientations (one launch per
    step, no amax)."""
    from nvfp4_block_scaled_quantize_gb300 import api, _lib
    _lib.load()
    dev = torch.device("cuda", local)
    w = workloads.WORKLOADS[args.workload]
    if w.grouped or w.block2d:
        raise SystemExit("--mx runs on plain 1D workloads")
    fmt = args.mx
    inp = workloads.make_input(w)
    x = inp["x"].to(dev)
    ideal = mx_ideal_bytes(w, fmt)
    stream = torch.cuda.current_stream(dev)
    alloc = lambda: api.alloc_mx_outputs(w.rows, w.cols, dev, fmt, w.rowwise, w.columnwise)
    out = alloc()
    n_sets, flush, l2_note = l2_plan(args, dev, nbytes(x, *out.values()))
    sets = [(x, out)] + [(x.clone(), alloc()) for _ in range(n_sets - 1)]

    def step(j):
        xj, oj = sets[j % n_sets]
        api.nvfp4_mx_quantize(xj, fmt, w.rowwise, w.columnwise, out=oj)

    # timed as in run_ours: back to back between one event pair with rotating sets, per-step
    # events (a separate pass) for the spread; per-step events in the timed region with the flush
    per_step_timed = args.l2 == "flush"
    n_ev = args.steps if per_step_timed else min(args.steps, 1000)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_ev)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index if dev.index is not None else 0) as clocks:
        time.sleep(0.3)
        for j in range(args.warmup):
            clear_l2(flush)
            step(j)
        torch.cuda.synchronize(dev)
        status, bits = api.nvfp4_get_status(dev)
        if status != 0:
            raise RuntimeError("device status %d (bits %#x) after warm-up" % (status, bits))
        barrier(world)
        torch.cuda.synchronize(dev)
        clocks.mark_start()
        if per_step_timed:
            for i in range(args.steps):
                clear_l2(flush)
                events[i][0].record(stream)
                step(args.warmup + i)
                events[i][1].record(stream)
        else:
            t_start.record(stream)
            for i in range(args.steps):
                step(args.warmup + i)
            t_end.record(stream)
        torch.cuda.synchronize(dev)
        clocks.mark_end()
        time.sleep(0.05)
    barrier(world)
    if not per_step_timed:
        for i in range(n_ev):
            events[i][0].record(stream)
            step(args.warmup + args.steps + i)
            events[i][1].record(stream)
        torch.cuda.synchronize(dev)
    step_ms = [e[0].elapsed_time(e[1]) for e in events]
    total_s = max_over_ranks(world, (sum(step_ms) if per_step_timed
                                     else t_start.elapsed_time(t_end)) / 1e3)
    value = aggregate_gbs(ideal, args.steps, world, total_s)

    # end to end: pinned host input -> device -> quantize -> pinned host outputs, one stream
    x_host = inp["x"].pin_memory()
    host_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in out.items()}
    h2d = x_host.numel() * 2
    d2h = sum(v.numel() for v in out.values())

    def e2e_step():
        xd = x_host.to(dev, non_blocking=True)
        o = api.nvfp4_mx_quantize(xd, fmt, w.rowwise, w.columnwise, out=out)
        for k, v in o.items():
            host_out[k].copy_(v, non_blocking=True)
    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize(dev)
    e2e_steps = min(args.steps, 100)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_s = max_over_ranks(world, e0.elapsed_time(e1) / 1e3)
    if rank != 0:
        return
    hbm, peak_kind = peaks()
    kus = total_s * 1e6 / args.steps  # one launch per step
    achieved = ideal / (kus / 1e6) / 1e9
    line = {
        "metric": MX_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_s * 1e3 / args.steps,
        "elements_per_s": w.rows * w.cols * args.steps * world / total_s,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "shape": [w.rows, w.cols], "format": "MX" + fmt,
                   "rowwise": w.rowwise, "columnwise": w.columnwise,
                   "ideal_bytes_per_step": ideal, "pipeline": "one launch (no amax)",
                   "l2": l2_note,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "gpu_launches": args.steps,
        "e2e": {"value": ideal * e2e_steps * world / e2e_s / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "path": "nvfp4_mx_quantize, copies on the current stream"},
        "clocks": clocks.summary(),
        "step_us": {"min": min(step_ms) * 1e3, "median": statistics.median(step_ms) * 1e3,
                    "max": max(step_ms) * 1e3},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "peak_kind": peak_kind,
                     "kernel": "mx_quantize_kernel", "kernel_us": kus, "traffic": None},
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = mx_cpu_baseline(w, inp, fmt)
    print(json.dumps(line), flush=True)


PRODUCER_METRIC = "RMSNorm + NVFP4 quantize GB/s (BF16 in) with the amax in the norm's epilogue, 1 GPU"


def run_producer(args, world, rank, local):
    """--producer rmsnorm: nvfp4_rmsnorm_quantize (the norm's epilogue gives the amax: norm +
    quantize, two launches) on the workload, timed beside the same norm followed by
    nvfp4_quantize computing its own amax in one launch (fused_amax)."""
    from nvfp4_block_scaled_quantize_gb300 import api, _lib
    _lib.load()
    dev = torch.device("cuda", local)
    w = workloads.WORKLOADS[args.workload]
    if w.grouped:
        raise SystemExit("--producer runs on plain workloads")
    inp = workloads.make_input(w)
    x = inp["x"].to(dev)
    kw = quant_kwargs(w, inp)
    weight = torch.ones(w.cols, dtype=torch.bfloat16, device=dev)
    alloc = lambda: api.alloc_outputs(w.rows, w.cols, dev, w.rowwise, w.columnwise)
    out = alloc()
    y = torch.empty_like(x)
    amax = torch.empty(1, dtype=torch.float32, device=dev)
    n = w.rows * w.cols
    # x read, y written and read back, plus the quantize outputs
    ideal = 2 * n + 2 * n + ideal_bytes(w)
    stream = torch.cuda.current_stream(dev)
    n_sets, flush, l2_note = l2_plan(args, dev, nbytes(x, y, *out.values()))
    sets = [(x, y, out)] + [(x.clone(), torch.empty_like(x), alloc()) for _ in range(n_sets - 1)]

    def fused(j):
        xj, yj, oj = sets[j % n_sets]
        api.nvfp4_rmsnorm_quantize(xj, weight, eps=1e-6, out=oj, y=yj, amax=amax, **kw)

    def unfused(j):
        xj, yj, oj = sets[j % n_sets]
        api.nvfp4_rmsnorm_amax(xj, weight, eps=1e-6, y=yj, amax=amax)
        api.nvfp4_quantize(yj, out=oj, fused_amax=True, **kw)

    def timed(fn, steps):
        """Per-step times in ms: per-step events with the flush; otherwise the steps run back
        to back between one event pair and every step gets the mean."""
        for j in range(args.warmup):
            clear_l2(flush)
            fn(j)
        torch.cuda.synchronize(dev)
        if args.l2 == "flush":
            ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
            for i in range(steps):
                clear_l2(flush)
                ev[i][0].record(stream)
                fn(args.warmup + i)
                ev[i][1].record(stream)
            torch.cuda.synchronize(dev)
            return [e[0].elapsed_time(e[1]) for e in ev]
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for i in range(steps):
            fn(args.warmup + i)
        a1.record(stream)
        torch.cuda.synchronize(dev)
        return [a0.elapsed_time(a1) / steps] * steps

    with ClockSampler(dev.index if dev.index is not None else 0) as clocks:
        time.sleep(0.3)
        barrier(world)
        clocks.mark_start()
        step_ms = timed(fused, args.steps)
        clocks.mark_end()
        base_ms = timed(unfused, args.steps)
    status, bits = api.nvfp4_get_status(dev)
    if status != 0:
        raise RuntimeError("device status %d (bits %#x)" % (status, bits))
    total_s = max_over_ranks(world, sum(step_ms) / 1e3)
    if rank != 0:
        return
    hbm, peak_kind = peaks()
    value = aggregate_gbs(ideal, args.steps, world, total_s)
    line = {
        "metric": PRODUCER_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_s * 1e3 / args.steps,
        "elements_per_s": w.rows * w.cols * args.steps * world / total_s,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "shape": [w.rows, w.cols], "ideal_bytes_per_step": ideal,
                   "pipeline": "nvfp4_rmsnorm_quantize: norm (amax in its epilogue) + quantize",
                   "l2": l2_note},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks.summary(),
        "step_us": {"min": min(step_ms) * 1e3, "median": statistics.median(step_ms) * 1e3,
                    "max": max(step_ms) * 1e3},
        "unfused_step_us": {"median": statistics.median(base_ms) * 1e3,
                            "what": "the same norm, then nvfp4_quantize computing its own amax "
                                    "(fused_amax, one launch)"},
        "roofline": {"bound": "hbm", "achieved": value, "peak": hbm, "unit": "GB/s",
                     "frac": value / hbm, "peak_kind": peak_kind, "traffic": None,
                     "kernel": "rmsnorm_amax_kernel + quantize_tiles_kernel (the step)"},
    }
    print(json.dumps(line), flush=True)


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5000)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(workloads.WORKLOADS))
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--rows", type=int, default=0,
                   help="a smaller case of the workload (its first ROWS rows' shape and "
                        "distribution; profiling captures), not a bench line")
    p.add_argument("--l2", choices=["rotate", "flush"], default="rotate",
                   help="between timed steps: rotate input/output sets totalling >= 3x L2 "
                        "(inputs larger than L2), or write a 256 MiB buffer before each step")
    p.add_argument("--pipeline", choices=["fused", "two_pass"], default="fused",
                   help="fused: amax and quantize in one launch; two_pass: amax kernel then "
                        "quantize kernel")
    p.add_argument("--mx", choices=["e4m3", "e5m2", "e2m1"], default=None,
                   help="time the MX quantizer (MXFP8 E4M3/E5M2, MXFP4) on the workload's shape")
    p.add_argument("--producer", choices=["rmsnorm"], default=None,
                   help="time the RMSNorm producer with the amax in its epilogue + quantize")
    p.add_argument("--fast-math", action="store_true",
                   help="the fast-math variant (approximate reciprocal; FP32 RHT columnwise)")
    args = p.parse_args()
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.mx:
        run_mx(args, world, rank, local)
    elif args.producer:
        run_producer(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
