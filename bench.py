"""Benchmark of libtpoverlap on GB300.

One step = one overlapped AG+GEMM call of the 4096^3 workload (tp = 4 simulated
ranks, X_r [1024, 4096], W [4096, 4096], bf16 in, Y [4096, 4096] bf16 out):
ring-order chunk producer, per-chunk release counters, counter-gated tcgen05
GEMM, rank-order epilogue, in one launch.  The block of K steps is repeated
back to back until the timed region lasts --timed-seconds (clock record with
>= 10 samples; the rate the power cap sustains), and the roofline fraction is
taken against the measured sustained bf16 peak (the burst fraction beside it).
The line also reports the same call in sequential mode (copy, then GEMM), the
GEMM alone, the producer alone, the host link's copy bound beside the
end-to-end rate, and the other workloads (row-parallel GEMM+AR, GEMM+RS, FP8
AG+GEMM, the allocation-free entry point) each with its own clock record.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tpo|reference]

With N > 1 (launched by torch.distributed.run) every rank runs an independent
replica on its own GPU: the simulated ranks live in one GPU's memory, so the
path has no exchange between GPUs ("replicas only"); value = work of all
ranks / slowest rank's time.
"""

from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from tensor_comm_gemm_gb300 import synth  # noqa: E402

METRIC = "overlapped AG+GEMM / GEMM+RS TFLOP/s on 1 GB300; % of dense tensor peak"
HEADLINE = 1  # the 4096^3 AG+GEMM workload
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0  # nominal dense ratio (4.5 / 2.25 PFLOP/s)
ROTATE = 3  # copies of the headline workload's buffers used round robin


def describe(idx):
    op, dt, tp, n, k, m, ch = synth.WORKLOAD_SHAPES[idx]
    if op == "ag":
        return "AG+GEMM %s tp=%d: X_r [%d,%d], W [%d,%d] -> Y [%d,%d] bf16" % (dt, tp, n // tp, k, m, k, n, m)
    if op == "rs":
        return "GEMM+RS bf16 tp=%d: X_r [%d,%d], W_r [%d,%d] -> %d blocks [%d,%d]" % (
            tp, n, k // tp, m, k // tp, tp, n // tp, m)
    return "row-parallel GEMM+AR bf16 tp=%d, %d row chunks: X_r [%d,%d], W_r [%d,%d] -> Y [%d,%d]" % (
        tp, ch, n, k // tp, m, k // tp, n, m)


def kernel_sha() -> str:
    """Hash of the kernel sources' code (comments and blank space removed);
    DRAM traffic figures taken with ncu are only reported while they still
    describe the kernel as built."""
    h = hashlib.sha256()
    for f in ("kernels.cu", "tpo_params.h"):
        with open(os.path.join(ROOT, "tensor_comm_gemm_gb300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)    # block comments
        src = re.sub(r"//[^\n]*", " ", src)                  # line comments
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class Clocks:
    """nvidia-smi sampling of SM clock, power and throttle reasons for the whole
    benchmark (one sampler, 50 ms period); each measured region keeps its host
    wall-clock window and gets its own record from the samples inside it."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.rows = None
        self.path = os.path.join("/tmp", "tpo_clocks_%d_%d.csv" % (os.getpid(), gpu_index))

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        if self.proc is not None:
            import atexit
            atexit.register(self._kill)   # never leave the sampler running past this process
        time.sleep(0.5)                # let the sampler come up before the first region

    def _kill(self):
        if self.proc is not None and self.proc.poll() is None:
            self.proc.kill()

    def stop(self):
        """Ends sampling and reads every sample (timestamp, clock, max clock,
        power, active throttle reasons)."""
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        import datetime
        self.rows = []
        with open(self.path) as f:
            for ln in f:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    clk, cmax = float(parts[1]), float(parts[2])
                except ValueError:
                    continue
                try:
                    pw = float(parts[3])
                except ValueError:
                    pw = None
                act = [nm for nm, v in zip(self.NAMES, parts[4:8]) if v.lower().startswith("active")]
                self.rows.append((ts, clk, cmax, pw, act))
        os.unlink(self.path)

    def window(self, t_begin, t_end, limits=False):
        """Median SM clock, maximum clock, throttle reasons and sample count of
        the samples taken between t_begin and t_end (host wall-clock seconds)."""
        if self.rows is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sel = [r for r in self.rows if t_begin - 0.05 <= r[0] <= t_end + 0.05]
        sm = [r[1] for r in sel]
        power = [r[3] for r in sel if r[3] is not None]
        out = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(r[2] for r in sel) if sel else None,
               "reasons": sorted({a for r in sel for a in r[4]}), "samples": len(sel),
               "power_w_max": max(power) if power else None, "window_s": round(t_end - t_begin, 3)}
        if limits:
            out["power_limits_w"] = self.power_limits()
        return out

    def power_limits(self):
        """The board's enforced and maximum power limits (read only)."""
        try:
            out = subprocess.run(["nvidia-smi", "-i", str(self.gpu),
                                  "--query-gpu=enforced.power.limit,power.max_limit",
                                  "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=10)
            enforced, mx = [float(v) for v in out.stdout.strip().split(",")[:2]]
            return {"enforced": enforced, "max": mx}
        except (OSError, ValueError, subprocess.TimeoutExpired):
            return None


# ---------------------------------------------------------------------------- aggregation

def slowest_rank_ms(ms, dist, device=None):
    """Per-step time of the slowest rank (every rank runs its own replica)."""
    if dist is None:
        return ms
    import torch
    tt = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def whole_job_tflops(flops_per_replica, world, ms):
    """Work of all ranks divided by the slowest rank's time."""
    return world * flops_per_replica / (ms * 1e-3) / 1e12


# ---------------------------------------------------------------------------- GPU arm

def gpu_arm(args, rank, world, local_rank, dist):
    import torch
    from tensor_comm_gemm_gb300 import build as tb
    from tensor_comm_gemm_gb300 import tpoverlap as t

    tb.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peaks, peak_kind = load_peaks()
    stream = torch.cuda.current_stream()
    clocks = Clocks(local_rank)          # one sampler for the whole run; regions keep their windows
    clocks.start()

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    def time_steps(fn, steps, warmup):
        """Per-step CUDA-event durations (ms) on the launching stream, steps back to
        back.  fn(i) runs step i; the events are created before the loop so that the
        host stays ahead of the GPU and no step waits for its own launch."""
        for i in range(warmup):
            fn(i)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(evs):
            a.record(stream)
            fn(i)
            b.record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    def time_row(fn, steps, warmup, seconds):
        """A measured row: warm-up, then back-to-back steps for at least `seconds`
        (and at least `steps` of them) in one timed region; returns (mean ms per
        step, the region's wall-clock window for its clock record, step count)."""
        probe = time_steps(fn, 2, warmup)
        count = max(steps, int(np.ceil(seconds * 1e3 / max(min(probe), 1e-3))))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0 = time.time()
        e0.record(stream)
        for i in range(count):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize()
        t1 = time.time()
        return e0.elapsed_time(e1) / count, (t0, t1), count

    def mean(v):
        return sum(v) / len(v)

    def check(ctx):
        st = t.tpo_sync_status(ctx)
        if st != 0:
            raise RuntimeError("device failure: " + t.tpo_last_error())

    # ---- headline workload: AG+GEMM tp=4, 4096^3
    wl = synth.workload(HEADLINE)
    flops = synth.flops(HEADLINE)
    # The workload's inputs and output (96 MiB) fit in the 129 MB L2, so the steps
    # rotate over ROTATE copies of X_r, W and Y (3 x 96 MiB): no step finds its
    # operands in L2 from the step before, and no flush kernel is needed.
    xs_sets = [[to_dev(x) for x in wl.x] for _ in range(ROTATE)]
    w_sets = [to_dev(wl.w[0]) for _ in range(ROTATE)]
    y_sets = [torch.empty((wl.n, wl.m), dtype=torch.bfloat16, device=dev) for _ in range(ROTATE)]
    xs, w, y = xs_sets[0], w_sets[0], y_sets[0]
    ctx = t.tpo_ctx_create(wl.tp, wl.n, wl.k, wl.m, t.TPO_BF16)
    if args.producer_sms:
        t.tpo_set_opt(ctx, "producer_sms", args.producer_sms)
    lib = t.lib()
    ptr_arrays = [t._ptr_array(xs_sets[j]) for j in range(ROTATE)]  # kept alive: the calls read them
    raw_args = [(t._addr(ptr_arrays[j]), w_sets[j].data_ptr(), y_sets[j].data_ptr()) for j in range(ROTATE)]
    sh = stream.cuda_stream

    def call(i=0):
        xa, wp, yp = raw_args[i % ROTATE]
        st = lib.tpo_ag_gemm(ctx, xa, wp, yp, None, None, sh)
        if st:
            raise t.TpoError(st, t.tpo_last_error())

    def mode_times(mode, steps, warmup):
        t.tpo_set_opt(ctx, "mode", mode)
        v = time_steps(call, steps, warmup)
        check(ctx)
        return v

    detail_steps = min(200, max(5, args.steps // 2))
    detail_t0 = time.time()
    seq = mode_times(1, detail_steps, 3)
    prod_only = mode_times(3, detail_steps, 3)
    split = mode_times(4, detail_steps, 3)
    # exposed producer time: overlapped and GEMM-only calls in interleaved blocks of
    # equal length, so that both see the same clock and power state
    ov_blocks, gemm_only = [], []
    for _ in range(4):
        ov_blocks += mode_times(0, detail_steps // 2 or 1, 2)
        gemm_only += mode_times(2, detail_steps // 2 or 1, 2)
    detail_t1 = time.time()
    t.tpo_set_opt(ctx, "mode", 0)

    # ---- the timed region: the block of K overlapped steps, repeated back to back
    # R times so that the region lasts at least --timed-seconds (the clock sampler's
    # 50 ms period then gives >= 10 samples, and the rate is the sustained one the
    # power cap allows), bracketed by a barrier + synchronize on both sides; the
    # per-step time is the mean over all R x K steps.
    for i in range(args.warmup):
        call(i)
    check(ctx)
    est_ms = min(mean(ov_blocks), mean(gemm_only))
    repeats = max(1, int(np.ceil(args.timed_seconds * 1e3 / (args.steps * est_ms))))
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("tpo_timed")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(repeats)]
    wall0 = time.time()
    t0 = time.perf_counter()
    for r, (a, b) in enumerate(evs):
        a.record(stream)
        for i in range(args.steps):
            call(r * args.steps + i)
        b.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    wall1 = time.time()
    torch.cuda.nvtx.range_pop()
    if dist is not None:
        dist.barrier()
    check(ctx)
    block_ms = [a.elapsed_time(b) for a, b in evs]
    step_ms = [bm / args.steps for bm in block_ms]
    ms = slowest_rank_ms(sum(block_ms) / (repeats * args.steps), dist, dev)
    value = whole_job_tflops(flops, world, ms)
    windows = {"headline": (wall0, wall1), "detail": (detail_t0, detail_t1)}

    # ---- the SM clock inside the kernel (GEMM CTAs' cycles per global-timer ns of the
    # kernel span, median of several traced calls); nvidia-smi's clocks.sm reading does
    # not show the clock the tensor cores run at.  CTAs that run out of tiles before the
    # last round ends stop counting early, so this reads somewhat low.
    t.tpo_set_opt(ctx, "trace", 1)
    mhz = []
    for _ in range(7):
        call()
        check(ctx)
        tr = t.tpo_read_trace(ctx)
        gemm_ctas = t.tpo_get_opt(ctx, "last_gemm_ctas")
        span_ns = max(1, tr[t.TPO_TRACE_END] - tr[t.TPO_TRACE_START])
        mhz.append(tr[t.TPO_TRACE_CYC_GEMM] / max(1, gemm_ctas) / span_ns * 1e3)
    t.tpo_set_opt(ctx, "trace", 0)
    sm_mhz_in_kernel = round(statistics.median(mhz), 0)

    # ---- end to end through the C ABI with host buffers.  Every step uploads its
    # activations X_r from pinned host memory and reads its result Y back; W is the
    # layer's weight and stays resident, as in a model.  Steps are double-buffered
    # on separate copy streams: step i+1's upload and step i-1's download overlap
    # step i's call, which is what a serving loop does.
    # The ranks' chunks sit back to back in one pinned host buffer and in one device
    # buffer per step, so each step uploads them with a single copy (the library
    # takes one pointer per rank: row slices of that buffer).
    rows = wl.n // wl.tp
    hx_all = torch.from_numpy(np.ascontiguousarray(np.concatenate(wl.x, 0)).view(np.int16)).view(
        torch.bfloat16).pin_memory()
    hy = [torch.empty((wl.n, wl.m), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dx_all = [torch.empty_like(hx_all, device=dev) for _ in range(2)]
    dx = [[d[r * rows:(r + 1) * rows] for r in range(wl.tp)] for d in dx_all]
    dy = [torch.empty_like(y) for _ in range(2)]
    s_up, s_down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731

    def e2e_run(steps):
        up = [ev(), ev()]
        done = [ev(), ev()]
        down = [ev(), ev()]
        t_a, t_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t_a.record(stream)
        s_up.wait_stream(stream)
        s_down.wait_stream(stream)
        for i in range(steps):
            j = i & 1
            if i >= 2:
                s_up.wait_event(done[j])        # step i-2 finished reading dx[j]
            with torch.cuda.stream(s_up):
                dx_all[j].copy_(hx_all, non_blocking=True)
                up[j].record(s_up)
            stream.wait_event(up[j])
            if i >= 2:
                stream.wait_event(down[j])      # dy[j] of step i-2 is back on the host
            t.tpo_ag_gemm(ctx, dx[j], w, dy[j], stream=stream)
            done[j].record(stream)
            s_down.wait_event(done[j])
            with torch.cuda.stream(s_down):
                hy[j].copy_(dy[j], non_blocking=True)
                down[j].record(s_down)
        stream.wait_stream(s_up)
        stream.wait_stream(s_down)
        t_b.record(stream)
        torch.cuda.synchronize()
        return t_a.elapsed_time(t_b) / steps

    e2e_run(3)
    e2e_ms = e2e_run(detail_steps)
    check(ctx)
    assert torch.equal(hy[(detail_steps - 1) & 1], y_sets[0].cpu()), "end-to-end result differs from the device run"
    h2d = sum(x.nbytes for x in wl.x)
    d2h = wl.n * wl.m * 2
    link = host_link(torch, dev, h2d, d2h)
    link["e2e_frac_of_copy_bound"] = round(link["copy_bound_ms"] / e2e_ms, 4)

    # ---- roofline of the dominant kernel (the fused launch) from the events above
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    achieved = flops / (sum(block_ms) / (repeats * args.steps) * 1e-3) / 1e12
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        with open(tpath) as f:
            tj = json.load(f)
        if tj.get("kernel_sha") == kernel_sha():
            traffic = tj.get("ag_tp4_4096", {}).get("bytes_per_launch")
    gemm_ms, seq_ms, prod_ms = mean(gemm_only), mean(seq), mean(prod_only)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    producer_bytes = 2 * (wl.n * wl.k * 2)  # every chunk read once and written once
    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded splitmix64 normal inputs, sigma = K^-1/4)",
        "config": {"workload": "ag_tp4_4096: " + describe(HEADLINE), "mode": "overlapped (one launch)",
                   "producer_ctas": t.tpo_get_opt(ctx, "last_producer_ctas"), "gemm_ctas": t.tpo_get_opt(ctx, "last_gemm_ctas"), "cta_group": t.tpo_get_opt(ctx, "last_cta_group"),
                   "stage_kblocks": t.tpo_get_opt(ctx, "last_stage_kblocks"),
                   "cooperative_launch": bool(t.tpo_get_opt(ctx, "cooperative") and t.tpo_get_opt(ctx, "coop_clusters")),
                   "programmatic_dependent_launch": bool(t.tpo_get_opt(ctx, "pdl")),
                   "l2": "inputs larger than L2: %d rotating sets of X_r, W, Y (%d MiB), steps back to back" % (
                       ROTATE, ROTATE * 96),
                   "parallelism": "replicas only (simulated ranks in one GPU's memory)"},
        "gpu_launches": repeats * args.steps,
        "timing": {"repeats": repeats, "steps_timed": repeats * args.steps,
                   "block_ms_min": round(min(block_ms), 5), "block_ms_max": round(max(block_ms), 5),
                   "note": "the K-step block run %d times back to back (>= %.1f s, sustained power state); "
                           "ms_per_step is the mean over all of them" % (repeats, args.timed_seconds)},
        "wall_s_timed_region": round(wall, 4),
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 5),
                "note": "per step: the X_r (one pinned host buffer, one copy) uploaded, Y read back; W "
                        "resident (layer weight); steps double-buffered on copy streams",
                "link": link},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak_sus, "unit": "TFLOP/s",
                     "frac": round(achieved / peak_sus, 4), "traffic": traffic,
                     "peak_source": ("%s bf16 sustained (MEASURED_PEAKS.json): the kernel is timed inside a "
                                     "%.1f s run of back-to-back steps" % (peak_kind, wall)) if peak_kind == "measured"
                     else "fallback 1.7 PFLOP/s sustained",
                     "peak_burst": peak, "frac_of_burst": round(achieved / peak, 4)},
        "detail": {
            "sequential_ms": round(seq_ms, 5),
            "sequential_tflops": round(flops / (seq_ms * 1e-3) / 1e12, 2),
            "gemm_only_ms": round(gemm_ms, 5),
            "gemm_only_tflops": round(flops / (gemm_ms * 1e-3) / 1e12, 2),
            "producer_only_ms": round(prod_ms, 5),
            "producer_only_gbs": round(producer_bytes / (prod_ms * 1e-3) / 1e9, 1),
            "producer_frac_of_hbm": round(producer_bytes / (prod_ms * 1e-3) / 1e9 / hbm, 4),
            "exposed_producer_frac": round((mean(ov_blocks) - gemm_ms) / gemm_ms, 4),
            "exposed_note": "overlapped vs GEMM-only (staging prefilled) in interleaved blocks",
            "split_ms": round(mean(split), 5),
            "split_tflops": round(flops / (mean(split) * 1e-3) / 1e12, 2),
        },
    }
    t.tpo_ctx_destroy(ctx)
    del xs, w, y, xs_sets, w_sets, y_sets, hx_all, hy, dx, dx_all, dy

    # ---- the other workloads, one line each inside "also"
    cpu_others = {} if (rank == 0 and not args.no_cpu) else None
    if not args.headline_only:
        result["also"] = other_workloads(args, dev, to_dev, time_steps, time_row, mean, peak, peak_sus, check, t,
                                         torch, cpu_others)

    # ---- clock records: the headline's timed region, the detail modes, and every
    # "also" row from its own window
    clocks.stop()
    clk = clocks.window(*windows["headline"], limits=True)
    clk["sm_mhz_in_kernel"] = sm_mhz_in_kernel
    result["clocks"] = clk
    result["roofline"]["nominal"] = nominal_peak(achieved, sms, clk.get("sm_max_mhz"), sm_mhz_in_kernel)
    result["detail"]["clocks"] = clocks.window(*windows["detail"])
    for rec in (result.get("also") or {}).values():
        if isinstance(rec, dict) and "_window" in rec:
            rec["clocks"] = clocks.window(*rec.pop("_window"))

    # ---- the oracle on the host cores, bounded sample
    if rank == 0 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds, cpu_others)
    return result


def host_link(torch, dev, h2d_bytes, d2h_bytes, reps=10):
    """The host link's own rate, for the end-to-end step's copy bound: one plain
    pinned-memory cudaMemcpyAsync of the step's upload size host to device, one
    of its download size device to host, each alone and both at once on two
    streams (mean of `reps` copies)."""
    hu = torch.empty(h2d_bytes, dtype=torch.uint8).pin_memory()
    du = torch.empty(h2d_bytes, dtype=torch.uint8, device=dev)
    hd = torch.empty(d2h_bytes, dtype=torch.uint8).pin_memory()
    dd = torch.empty(d2h_bytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def timed(fn):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / reps

    def up():
        with torch.cuda.stream(s1):
            du.copy_(hu, non_blocking=True)

    def down():
        with torch.cuda.stream(s2):
            hd.copy_(dd, non_blocking=True)

    def both():
        up()
        down()
    t_up, t_down, t_both = timed(up), timed(down), timed(both)
    bound_s = max(h2d_bytes / (h2d_bytes / t_up), d2h_bytes / (d2h_bytes / t_down), t_both)
    return {"h2d_gbs": round(h2d_bytes / t_up / 1e9, 1), "d2h_gbs": round(d2h_bytes / t_down / 1e9, 1),
            "both_directions_gbs": round((h2d_bytes + d2h_bytes) / t_both / 1e9, 1),
            "copy_bound_ms": round(bound_s * 1e3, 5),
            "note": "one pinned cudaMemcpyAsync of the step's upload and one of its download, alone and "
                    "together; copy_bound_ms = the slower of the two alone or both at once"}


def nominal_peak(achieved, sms, max_mhz, kernel_mhz):
    """The tensor rate from the hardware's unit count: SMs x 8192 bf16 FLOP per
    clock per SM (an assumption, the figure ncu gives as peak_sustained), at the
    maximum SM clock and at the clock measured inside the kernel."""
    out = {"flop_per_clk_per_sm": 8192, "sms": sms}
    for key, mhz in (("max_clock", max_mhz), ("kernel_clock", kernel_mhz)):
        if mhz:
            pk = sms * 8192 * mhz * 1e6 / 1e12
            out["peak_at_" + key] = round(pk, 1)
            out["frac_at_" + key] = round(achieved / pk, 4)
    return out


def cublas_fp8_tflops(torch, dev, size=8192):
    """Dense e4m3 GEMM rate of the vendor library (torch._scaled_mm, size^3), the
    measured FP8 counterpart of the bf16 peak; None where the call is missing."""
    try:
        a = torch.randn(size, size, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(size, size, device=dev).to(torch.float8_e4m3fn)
        one = torch.ones((), device=dev)
        f = lambda: torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)  # noqa: E731
        for _ in range(3):
            f()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(10):
            f()
        e1.record()
        torch.cuda.synchronize()
        return round(2.0 * size ** 3 / (e0.elapsed_time(e1) / 10 * 1e-3) / 1e12, 1)
    except Exception:  # noqa: BLE001
        return None


def library_gemm_4096(torch, dev, sets=3, calls=60):
    """The vendor library's plain bf16 GEMM (torch.matmul) on the headline's
    4096^3 shape, rotating over input sets as the headline does: the GEMM alone,
    with no chunk movement, for context beside the overlapped call."""
    try:
        xs = [torch.randn(4096, 4096, device=dev, dtype=torch.bfloat16) for _ in range(sets)]
        ws = [torch.randn(4096, 4096, device=dev, dtype=torch.bfloat16) for _ in range(sets)]
        ys = [torch.empty(4096, 4096, device=dev, dtype=torch.bfloat16) for _ in range(sets)]
        for i in range(6):
            torch.matmul(xs[i % sets], ws[i % sets].t(), out=ys[i % sets])
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for i in range(calls):
            torch.matmul(xs[i % sets], ws[i % sets].t(), out=ys[i % sets])
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / calls
        return {"ms": round(ms, 5), "tflops": round(2.0 * 4096 ** 3 / (ms * 1e-3) / 1e12, 1)}
    except Exception:  # noqa: BLE001
        return None


def other_workloads(args, dev, to_dev, time_steps, time_row, mean, peak, peak_sus, check, t, torch,
                    cpu_others=None):
    """One record per other workload.  Each tensor-bound row times at least
    args.row_seconds of back-to-back steps and keeps that window for its own
    clock record; its rate is given against the sustained and the burst
    measured peak (FP8 rows: twice each, the nominal dense ratio)."""
    out = {}
    steps = min(40, max(5, args.steps // 2))
    # the small AG workload: latency-bound (a few output tiles), reported in microseconds per call of
    # back-to-back calls (one event pair around the whole run, so no per-call event joins the timing)
    wl = synth.workload(0)
    xs = [to_dev(x) for x in wl.x]
    w = to_dev(wl.w[0])
    y = torch.empty((wl.n, wl.m), dtype=torch.bfloat16, device=dev)
    ctx = t.tpo_ctx_create(wl.tp, wl.n, wl.k, wl.m, t.TPO_BF16)
    lib, xarr, sh = t.lib(), t._ptr_array(xs), torch.cuda.current_stream().cuda_stream
    xa = t._addr(xarr)

    def raw(i=0):
        st = lib.tpo_ag_gemm(ctx, xa, w.data_ptr(), y.data_ptr(), None, None, sh)
        if st:
            raise t.TpoError(st, t.tpo_last_error())
    t0 = time.time()
    ms = time_row(raw, 2000, 20, 0.02)[0]
    ms_py = time_row(lambda i=0: t.tpo_ag_gemm(ctx, xs, w, y), 2000, 20, 0.02)[0]
    check(ctx)
    # us_per_call: the C ABI call; us_per_call_python adds the binding's argument checks
    out[wl.name] = {"workload": describe(0), "us_per_call": round(ms * 1e3, 2),
                    "us_per_call_python": round(ms_py * 1e3, 2),
                    "tflops": round(synth.flops(0) / (ms * 1e-3) / 1e12, 3), "_window": (t0, time.time())}
    if cpu_others is not None:   # small enough for the oracle to run in full
        cpu_others[wl.name] = oracle_full(wl)
    t.tpo_ctx_destroy(ctx)
    out["library_bf16_gemm_4096"] = library_gemm_4096(torch, dev)
    fp8_lib = cublas_fp8_tflops(torch, dev)
    out["fp8_library_gemm_8192"] = {"tflops": fp8_lib, "note": "torch._scaled_mm e4m3 8192^3 burst on this "
                                    "box; the FP8 rows' frac_of_peak uses 2 x the measured bf16 peak"}
    out["ag_tp4_4096_noalloc"] = noalloc_row(t, torch, dev, to_dev, peak)

    def rates(flops, ms, pk, pk_sus):
        """Rate against the sustained measured peak (the row is timed over a long
        back-to-back run) and against the burst peak."""
        tf = flops / (ms * 1e-3) / 1e12
        return {"tflops": round(tf, 2), "frac_of_peak": round(tf / pk_sus, 4), "peak_tflops": pk_sus,
                "peak_kind": "sustained", "frac_of_burst_peak": round(tf / pk, 4), "burst_peak_tflops": pk}

    for idx in (2, 3, 4):
        op, dt, tp, n, k, m, ch = synth.WORKLOAD_SHAPES[idx]
        wl = synth.workload(idx)
        flops = synth.flops(idx)
        name = wl.name
        if op == "ag":
            xs = [to_dev(x) for x in wl.x]
            w = to_dev(wl.w[0])
            y = torch.empty((n, m), dtype=torch.bfloat16, device=dev)
            sx = torch.tensor([wl.scale_inv_x], dtype=torch.float32, device=dev)
            sw = torch.tensor([wl.scale_inv_w], dtype=torch.float32, device=dev)
            ctx = t.tpo_ctx_create(tp, n, k, m, t.TPO_FP8_E4M3)
            fn = lambda i=0: t.tpo_ag_gemm(ctx, xs, w, y, sx, sw)  # noqa: E731
            pk, pk_sus = peak * FP8_OVER_BF16, peak_sus * FP8_OVER_BF16
        else:
            xs = [to_dev(x) for x in wl.x]
            ws = [to_dev(x) for x in wl.w]
            ctx = t.tpo_ctx_create(tp, n, k, m, t.TPO_BF16)
            if op == "rs":
                yb = [torch.empty((n // tp, m), dtype=torch.bfloat16, device=dev) for _ in range(tp)]
                fn = lambda i=0: t.tpo_gemm_rs(ctx, xs, ws, yb)  # noqa: E731
            else:
                y = torch.empty((n, m), dtype=torch.bfloat16, device=dev)
                fn = lambda i=0: t.tpo_gemm_ar(ctx, xs, ws, y, ch)  # noqa: E731
            pk, pk_sus = peak, peak_sus
        ms, window, count = time_row(fn, steps, 3, args.row_seconds)
        check(ctx)
        rec = {"workload": describe(idx), "ms": round(ms, 4), "steps_timed": count}
        rec.update(rates(flops, ms, pk, pk_sus))
        rec["_window"] = window
        if dt == "e4m3" and fp8_lib:
            rec["frac_of_library_fp8"] = round(flops / (ms * 1e-3) / 1e12 / fp8_lib, 4)
        if cpu_others is not None:  # the CPU-baseline leg: the oracle on a sample of this workload
            cpu_others[name] = other_sample(wl, max(1.0, args.cpu_seconds / 4))
        if op in ("rs", "ar"):
            # when each output group (RS owner block, AR row chunk) was complete, as a
            # fraction of the call: the point at which its communication could start
            t.tpo_set_opt(ctx, "trace", 1)
            fn()
            check(ctx)
            tr = t.tpo_read_trace(ctx)
            t.tpo_set_opt(ctx, "trace", 0)
            span = max(1, tr[t.TPO_TRACE_END] - tr[t.TPO_TRACE_START])
            groups = tp if op == "rs" else ch
            rec["group_done_frac"] = [round((tr[t.TPO_TRACE_CHUNK_DONE + gi] - tr[t.TPO_TRACE_START]) / span, 3)
                                      for gi in range(groups)]
        if op == "rs":  # the same call with the ranks' partials added in the epilogue
            for rmode, key in ((1, "epilogue_fp32"), (2, "epilogue_bf16_wire")):
                t.tpo_set_opt(ctx, "reduce", rmode)
                rms = mean(time_steps(fn, steps, 2))
                check(ctx)
                rec["reduce_" + key + "_ms"] = round(rms, 4)
            t.tpo_set_opt(ctx, "reduce", 0)
        if op == "ag":
            # overlapped, sequential and GEMM-only calls in interleaved short blocks, so
            # that the exposed producer time compares like with like (the sustained
            # rate above runs under the power cap, short blocks mostly do not)
            blk = {0: [], 1: [], 2: []}
            for _ in range(4):
                for mode in (0, 1, 2):
                    t.tpo_set_opt(ctx, "mode", mode)
                    blk[mode] += time_steps(fn, max(2, steps // 4), 1)
            t.tpo_set_opt(ctx, "mode", 0)
            check(ctx)
            ov, sms, gms = mean(blk[0]), mean(blk[1]), mean(blk[2])
            rec.update({"overlapped_ms_short_blocks": round(ov, 4), "sequential_ms": round(sms, 4),
                        "gemm_only_ms": round(gms, 4), "exposed_producer_frac": round((ov - gms) / gms, 4),
                        "exposed_note": "overlapped vs GEMM-only (staging prefilled) in interleaved short blocks"})
        out[name] = rec
        t.tpo_ctx_destroy(ctx)
        del fn
        torch.cuda.empty_cache()
    # the GEMM+RS down-projection shape with e4m3 K-slices (one scale for all X_r, one for all W_r)
    wl = synth.make_ksplit("rs", 8, 16384, 28672, 8192, seed=5, dtype="e4m3", name="rs_fp8_tp8_16384x8192x28672")
    xs = [to_dev(x) for x in wl.x]
    ws = [to_dev(x) for x in wl.w]
    yb = [torch.empty((wl.n // wl.tp, wl.m), dtype=torch.bfloat16, device=dev) for _ in range(wl.tp)]
    sx = torch.tensor([wl.scale_inv_x], dtype=torch.float32, device=dev)
    sw = torch.tensor([wl.scale_inv_w], dtype=torch.float32, device=dev)
    ctx = t.tpo_ctx_create(wl.tp, wl.n, wl.k, wl.m, t.TPO_FP8_E4M3)
    t.tpo_set_fp8_scales(ctx, sx, sw)
    ms, window, count = time_row(lambda i=0: t.tpo_gemm_rs(ctx, xs, ws, yb), steps, 3, args.row_seconds)
    check(ctx)
    flops = 2.0 * wl.n * wl.k * wl.m
    rec = {"workload": "GEMM+RS e4m3 tp=8: X_r [16384,3584], W_r [8192,3584] -> 8 blocks [2048,8192]",
           "ms": round(ms, 4), "steps_timed": count}
    rec.update(rates(flops, ms, peak * FP8_OVER_BF16, peak_sus * FP8_OVER_BF16))
    rec["_window"] = window
    if fp8_lib:
        rec["frac_of_library_fp8"] = round(flops / (ms * 1e-3) / 1e12 / fp8_lib, 4)
    out[wl.name] = rec
    t.tpo_ctx_destroy(ctx)
    return out


def noalloc_row(t, torch, dev, to_dev, peak, calls=50):
    """The allocation-free AG entry point on the 4096^3 workload beside the
    context call.  It returns only once its work is done (it reads the error
    word back), so a call's time is the host's wall time around it."""
    wl = synth.workload(HEADLINE)
    xs = [to_dev(x) for x in wl.x]
    w = to_dev(wl.w[0])
    y = torch.empty((wl.n, wl.m), dtype=torch.bfloat16, device=dev)
    for _ in range(3):
        t.tpo_ag_gemm_noalloc(wl.tp, wl.n, wl.k, wl.m, t.TPO_BF16, xs, w, y)
    torch.cuda.synchronize()
    times = []
    for _ in range(calls):
        t0 = time.perf_counter()
        t.tpo_ag_gemm_noalloc(wl.tp, wl.n, wl.k, wl.m, t.TPO_BF16, xs, w, y)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.median(times)
    tf = synth.flops(HEADLINE) / (ms * 1e-3) / 1e12
    return {"workload": describe(HEADLINE), "ms_per_call_median": round(ms, 4), "tflops": round(tf, 2),
            "frac_of_peak": round(tf / peak, 4), "peak_kind": "burst",
            "note": "tpo_ag_gemm_noalloc: default launch shape (CTA pairs, modelled producer count), blocking call (host wall "
                    "time per call, median of %d, includes the launch and the read-back of the error word)" % calls}


# ---------------------------------------------------------------------------- CPU oracle

def oracle_sample(wl, seconds, nthreads=None, seed=None):
    """The oracle as it stands over a bounded sample of the workload's 16 x 16
    output tiles (about `seconds` of work): (tiles timed, seconds, total tiles,
    FLOP per tile)."""
    import oracle

    tile = 16
    if wl.op == "ag":
        g = oracle.gather(wl.x)

        def run(tl):
            oracle.ag(g, wl.w[0], wl.scale_inv_x, wl.scale_inv_w, tiles=tl, nthreads=nthreads)
    else:
        def run(tl):
            oracle.ksplit(wl.x, wl.w, tiles=tl, nthreads=nthreads, sx=wl.scale_inv_x, sw=wl.scale_inv_w)
    probe = synth.sample_tiles(wl.n, wl.m, tile, 16, seed=7)
    t0 = time.perf_counter()
    run(probe)
    rate = len(probe) / max(time.perf_counter() - t0, 1e-6)
    count = int(max(16, min(65536, rate * seconds)))
    tiles = synth.sample_tiles(wl.n, wl.m, tile, count, seed=(1000 + wl.seed) if seed is None else seed)
    t0 = time.perf_counter()
    run(tiles)
    dt = time.perf_counter() - t0
    return len(tiles), dt, (wl.n // tile) * (wl.m // tile), 2.0 * tile * tile * wl.k


def cpu_baseline(wl, seconds, others=None):
    """The oracle as it stands, on the host cores, over a bounded sample of the
    workload's output tiles (16 x 16 each); throughput scaled to TFLOP/s.  Also:
    one core, the full problem's time extrapolated from the sample, and the
    same for the other workloads (`others`: name -> sampled record)."""
    import oracle

    n, dt, total, per_tile = oracle_sample(wl, seconds)
    n1, dt1, _, _ = oracle_sample(wl, max(1.0, seconds / 5), nthreads=1, seed=2000 + wl.seed)
    out = {"value": per_tile * n / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.threads(), "kind": "oracle",
           "sample": "%d of %d output tiles of 16x16 (FP64 loops over k=%d), %.1f s" % (n, total, wl.k, dt),
           "full_problem_s_extrapolated": round(dt * total / n, 1),
           "single_core": {"value": per_tile * n1 / dt1 / 1e12, "unit": "TFLOP/s", "cores": 1,
                           "sample": "%d output tiles, %.1f s" % (n1, dt1)}}
    if others:
        out["other_workloads"] = others
    return out


def oracle_full(wl, reps=5):
    """The oracle on the whole problem of a small workload (all host cores),
    the fastest of `reps` runs."""
    import oracle

    g = oracle.gather(wl.x)
    best = None
    for _ in range(reps):
        t0 = time.perf_counter()
        oracle.ag(g, wl.w[0], wl.scale_inv_x, wl.scale_inv_w)
        dt = time.perf_counter() - t0
        best = dt if best is None else min(best, dt)
    flops = 2.0 * wl.n * wl.k * wl.m
    return {"value": flops / best / 1e12, "unit": "TFLOP/s", "cores": oracle.threads(),
            "sample": "the full problem (%d x %d output, FP64 loops over k=%d), fastest of %d runs" % (
                wl.n, wl.m, wl.k, reps),
            "full_problem_s": round(best, 5)}


def other_sample(wl, seconds):
    """cpu_baseline's record of another workload: the oracle on a bounded
    sample of its output tiles, all host cores."""
    import oracle

    n, dt, total, per_tile = oracle_sample(wl, seconds)
    return {"value": per_tile * n / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.threads(),
            "sample": "%d of %d output tiles of 16x16 (FP64 loops over k=%d), %.1f s" % (n, total, wl.k, dt),
            "full_problem_s_extrapolated": round(dt * total / n, 1)}


def reference_arm(args):
    """The oracle timed as the reference arm: every step is a bounded sample of
    the headline workload's output tiles."""
    import oracle

    wl = synth.workload(HEADLINE)
    g = oracle.gather(wl.x)
    tile = 16
    per_tile = 2.0 * tile * tile * wl.k
    per_step = args.reference_seconds / max(1, args.steps + args.warmup)
    probe = synth.sample_tiles(wl.n, wl.m, tile, 16, seed=7)
    t0 = time.perf_counter()
    oracle.ag(g, wl.w[0], tiles=probe)
    rate = len(probe) / max(time.perf_counter() - t0, 1e-6)
    count = int(max(16, min(65536, rate * per_step)))
    times = []
    for i in range(args.warmup + args.steps):
        tiles = synth.sample_tiles(wl.n, wl.m, tile, count, seed=2000 + i)
        t0 = time.perf_counter()
        oracle.ag(g, wl.w[0], tiles=tiles)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = per_tile * count / (ms * 1e-3) / 1e12
    sample = "%d of %d output tiles of 16x16 per step (FP64 loops over k=%d)" % (
        count, (wl.n // tile) * (wl.m // tile), wl.k)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "ag_tp4_4096: " + describe(HEADLINE), "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="tpo", choices=["tpo", "reference"])
    ap.add_argument("--producer-sms", type=int, default=0)
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--timed-seconds", type=float, default=0.6,
                    help="shortest timed region: the K-step block is repeated until it lasts this long")
    ap.add_argument("--row-seconds", type=float, default=0.6,
                    help="shortest timed region of each other workload")
    ap.add_argument("--reference-seconds", type=float, default=90.0,
                    help="oracle work for the whole reference-arm run (split over its steps)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(reference_arm(args)), flush=True)
        return

    dist = None
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = gpu_arm(args, rank, world, local_rank, dist)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
