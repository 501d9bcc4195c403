#!/usr/bin/env python
"""Benchmark of the tile-level GEMM C = A * B on GB300.

One step is one C = A * B of the benchmark workload (default: M = N = K =
4096, bf16 inputs drawn from N(0, 1), fp32 accumulation, bf16 output) on
inputs already resident in HBM.  Between steps the L2 cache (129 MB) is
flushed by a read-only sweep of a 256 MB buffer (a sum into one scalar): the
sweep evicts the previous step's lines, including the dirty lines of its
output, and leaves none dirty, so no write-back of earlier data falls into a
timed step.  Each step's GEMM is timed with CUDA events on the launching
stream.

Prints one JSON line.  `value` is TFLOP/s (2*M*N*K per step) over all ranks;
`e2e` is the same metric through the same C ABI call with pinned host
buffers, the host->device copies of A and B and the device->host copy of C
inside the timed region; `roofline` relates the kernel to the measured bf16
tensor peak (for 8-bit inputs: twice that, the nominal fp8 : bf16 ratio),
or, below the ridge, to the measured HBM copy bandwidth; `cpu_baseline` is
the fp64 oracle timed on the host cores.  `workloads` holds the same
measurement (time per step, roofline, clocks, a sampled parity check) for
every other benchmark configuration and the 8-bit workloads, each timed
over the same number of steps after the headline.  --workload picks another
headline workload.

With --impl reference the fp64 CPU oracle itself is timed on the same
metric (a bounded sample of rows of the product per step).

Launch: python bench.py [--gpus N --steps K --warmup W]; for N > 1 under
torch.distributed.run, one rank per GPU, each running its own independent
instance of the workload (weak scaling, no data-path collective).
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "gemm_4096_bf16"
METRIC = "GEMM TFLOP/s and % of GB300 dense BF16 peak (4096^3; 16384x16384x8192)"
FLUSH_BYTES = 256 << 20
FALLBACK_BF16_TFLOPS = 1900.0

# Every workload timed after the headline one: the five benchmark
# configurations and the 8-bit workloads.
EXTRA_DEFAULT = ["gemm_256_f16_f32", "gemm_4096_bf16", "skinny_128x28672x8192_bf16",
                 "gemm_16384x16384x8192_bf16", "longk_1024x1024x65536_int_f32",
                 "gemm_4096_e4m3_rcr", "gemm_16384x16384x8192_e4m3_rcr"]
# nominal dense fp8 : bf16 tensor throughput on GB300 (4.5 : 2.25 PFLOP/s)
FP8_TO_BF16 = 2.0


def to_device_bits(bits, din, device=None, pin=False):
    """A torch tensor of the input format holding the numpy bit patterns."""
    import numpy as np
    import torch
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn,
           "e5m2": torch.float8_e5m2}[din]
    raw = np.ascontiguousarray(bits)
    t = torch.from_numpy(raw.view(np.uint8) if raw.dtype == np.uint8 else raw.view(np.int16))
    if pin:
        t = t.pin_memory()
    elif device is not None:
        t = t.to(device)
    return t.view(tdt)


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=0, help="default: min(steps, 50)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--plan", default="",
                    help="force plan fields of the headline workload, e.g. block_m=256,block_n=128,splits=1")
    ap.add_argument("--workloads", default="all",
                    help="workloads timed after the headline: 'all' (every benchmark configuration and "
                         "the 8-bit workloads), 'none', or a comma-separated list")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.steps < 1:
        ap.error("--steps must be at least 1")
    return args


# ----------------------------------------------------------- rank logic --

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed_offset(rank):
    """Each rank runs an independent instance of the workload: its seeds are
    the workload's seeds plus this offset."""
    return 0x10000 * rank


def max_over_ranks(x, world, device=None):
    """Largest value of x over all ranks (x on every rank)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(flops_per_step, ms_per_step_max, world):
    """Whole-job TFLOP/s: every rank did one step of flops_per_step in at most
    ms_per_step_max."""
    return world * flops_per_step / (ms_per_step_max * 1e-3) / 1e12


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.samples.append((time.time(), parts))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        return self.summary()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        inside = self.samples
        if self.window:
            t0, t1 = self.window
            w = [s for s in self.samples if t0 - 0.06 <= s[0] <= t1 + 0.06]
            if w:
                inside = w
        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(p[1]) for _, p in inside if num(p[1]) is not None]
        smax = [num(p[2]) for _, p in inside if num(p[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, p in inside:
            for name, v in zip(names, p[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(inside),
                "power_w_max": max((num(p[3]) or 0.0) for _, p in inside)}


# ----------------------------------------------------------------- peaks --

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return {"bf16_tflops": FALLBACK_BF16_TFLOPS, "hbm_gbs": 6800.0}, "fallback"


def bf16_peak(clocks):
    """The bf16 denominator and its description: the burst figure for a
    run at full clock, the sustained one when the sampled clocks show the
    power cap holding the SM clock well below its maximum (a long run of a
    large GEMM, the regime the sustained figure was measured in)."""
    peaks, kind = measured_peaks()
    capped = bool(clocks) and "sw_power_cap" in clocks.get("reasons", []) and \
        clocks.get("sm_mhz", 0) < 0.95 * clocks.get("sm_max_mhz", 1)
    if capped and "bf16_tflops_sustained" in peaks:
        return float(peaks["bf16_tflops_sustained"]), kind + " bf16 sustained (cuBLAS-class torch.matmul under the power cap)"
    return float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS)), kind + " bf16 burst (cuBLAS-class torch.matmul)"


def roofline_point(flops, algo_bytes, ms, tensor_peak, tensor_desc):
    """(bound, achieved, peak, unit, description) of a kernel that does
    `flops` and moves `algo_bytes` in `ms`: below the ridge (tensor peak /
    HBM bandwidth) it is bound by streaming its operands and is reported in
    GB/s against the measured HBM copy rate, else in TFLOP/s against
    `tensor_peak`."""
    peaks, kind = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    if flops / algo_bytes < tensor_peak * 1e12 / (hbm_peak * 1e9):
        return "hbm", algo_bytes / (ms * 1e-3) / 1e9, hbm_peak, "GB/s", kind + " HBM copy bandwidth"
    return "tensor", flops / (ms * 1e-3) / 1e12, tensor_peak, "TFLOP/s", tensor_desc


def kernel_sources():
    """Every file the library is built from (kernels, launch code, planner,
    instantiation tables, headers): a change to any of them may change a
    kernel's schedule and so its DRAM traffic."""
    import glob
    files = glob.glob(os.path.join(ROOT, "hierarchical_gemm_gb300", "csrc", "*"))
    files += glob.glob(os.path.join(ROOT, "include", "*.h"))
    return sorted(os.path.relpath(f, ROOT) for f in files if os.path.isfile(f))


def kernel_source_hash():
    h = hashlib.sha256()
    for rel in kernel_sources():
        h.update(rel.encode())
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def stored_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    with the current library source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(workload)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------- CPU oracle --

def oracle_rows_tflops(A, B, din, target_s, max_rows=None):
    """Time the fp64 oracle on the first R rows of the product, R grown until
    one evaluation takes about target_s seconds.  Returns (tflops, rows,
    seconds, threads)."""
    import numpy as np
    import oracle
    M, K = A.shape
    N = B.shape[1]
    max_rows = max_rows or M
    rows = min(8, max_rows)
    while True:
        t0 = time.perf_counter()
        _, _, used = oracle.gemm(np.ascontiguousarray(A[:rows]), B, din)
        dt = time.perf_counter() - t0
        if dt >= target_s * 0.5 or rows >= max_rows:
            return 2.0 * rows * N * K / dt / 1e12, rows, dt, used
        rows = min(max_rows, max(rows + 1, int(rows * target_s / max(dt, 1e-3))))


# ------------------------------------------------------------ reference --

def run_reference(args):
    """The oracle timed as the reference arm: every step evaluates a bounded
    sample of rows of the workload's product on the host cores."""
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import numpy as np
    import oracle
    import synth
    w = synth.workload(args.workload)
    A, B = synth.inputs(args.workload)  # logical A (M x K), B (K x N)
    # size one step at ~ (cpu_seconds / steps), at least 8 rows
    per_step = max(0.5, args.cpu_seconds / max(1, args.steps + args.warmup))
    _, rows, _, _ = oracle_rows_tflops(A, B, w["dtype_in"], per_step)
    Ar = np.ascontiguousarray(A[:rows])
    for _ in range(args.warmup):
        oracle.gemm(Ar, B, w["dtype_in"])
    t0 = time.perf_counter()
    used = 0
    for _ in range(args.steps):
        _, _, used = oracle.gemm(Ar, B, w["dtype_in"])
    dt = (time.perf_counter() - t0) / args.steps
    flops = 2.0 * rows * w["N"] * w["K"]
    value = flops / dt / 1e12
    sample = "rows 0..%d of the %dx%dx%d product per step" % (rows - 1, w["M"], w["N"], w["K"])
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": gemm_config(w, 1),
        "sample_rows": rows,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": used, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


# ------------------------------------------------------------------ ours --

class L2Sweep:
    """Read-only L2 flush: a sum of a 256 MB buffer (about twice the L2)
    into one scalar.  Reading evicts every line the previous step left in
    L2, dirty ones included (their write-back happens here, outside the
    timed region), and writes nothing but the scalar."""

    def __init__(self, dev):
        import torch
        self.buf = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        import torch
        torch.sum(self.buf, dim=0, out=self.sink)


def time_plan(plan, A, B, C, steps, warmup, dev, stream, flush, sampler_gpu, world):
    """Warm up, then time `steps` launches of the plan (each after an L2
    sweep) with CUDA events on the launching stream.  Returns (ms per step,
    max over ranks; clock summary or None)."""
    import torch
    from hierarchical_gemm_gb300 import tsgemm
    for _ in range(warmup):
        flush()
        plan.run(A, B, C, stream)
    torch.cuda.synchronize(dev)
    st = plan.status()
    if st != 0:
        raise RuntimeError("device status %d (%s) after warm-up" % (st, tsgemm.status_string(st)))
    sampler = ClockSampler(sampler_gpu) if sampler_gpu is not None else None
    if sampler:
        sampler.start()
        time.sleep(0.25)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    for i in range(steps):
        flush()
        starts[i].record(stream)
        plan.run(A, B, C, stream)
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    t_wall1 = time.time()
    clocks = None
    if sampler:
        sampler.mark(t_wall0, t_wall1)
        clocks = sampler.stop()
    st = plan.status()
    if st != 0:
        raise RuntimeError("device status %d (%s)" % (st, tsgemm.status_string(st)))
    ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / steps
    return max_over_ranks(ms, world, dev), clocks


def sampled_parity(C, A_np, B_np, w, count=1024, seed=7):
    """The oracle at `count` random outputs of this run's C."""
    import torch
    import oracle
    M, N = w["M"], w["N"]
    r = np.random.default_rng(seed)
    rows = r.integers(0, M, count)
    cols = r.integers(0, N, count)
    Ch = C.cpu()
    Ch = Ch.numpy() if w["dtype_out"] == "f32" else Ch.view(torch.int16).numpy().view(np.uint16)
    ref, sabs = oracle.gemm_sampled(A_np, B_np, w["dtype_in"], rows, cols)
    ok, info = oracle.accept(Ch[rows, cols], ref, sabs, w["dtype_out"], exact=w["exact"])
    return {"sampled_outputs": int(count), "ok": bool(ok), "exact": bool(w["exact"]),
            "max_err_over_bound": info.get("max_err_over_bound"), "mismatches": info.get("mismatches")}


def gemm_roofline(w, ms, clocks, cfg):
    """The roofline object of one GEMM workload timed at `ms` per launch."""
    import synth
    M, N, K = w["M"], w["N"], w["K"]
    din, dout = w["dtype_in"], w["dtype_out"]
    flops = 2.0 * M * N * K
    peak, peak_desc = bf16_peak(clocks)
    eight_bit = din in ("e4m3", "e5m2")
    if eight_bit:
        peak *= FP8_TO_BF16
        peak_desc += " x %.0f (nominal fp8 : bf16 dense ratio)" % FP8_TO_BF16
    algo_bytes = synth.workloads.in_nbytes(din) * (M * K + K * N) + synth.workloads.out_nbytes(dout) * M * N
    bound, achieved, peak, unit, peak_desc = roofline_point(flops, algo_bytes, ms, peak, peak_desc)
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": stored_traffic(w["name"]),
            "peak_kind": peak_desc,
            "kernel": "gemm_sm103_%s<BN=%d%s>" % ("2sm" if cfg["block_m"] == 256 else "1sm", cfg["block_n"],
                                                 ", 8-bit" if eight_bit else ""),
            "algorithmic_flops_per_launch": flops,
            "algorithmic_bytes_per_launch": algo_bytes}


def gemm_config(w, world):
    """The `config` object of a GEMM workload's line (the same for both
    arms of the benchmark)."""
    return {"workload": w["name"], "M": w["M"], "N": w["N"], "K": w["K"], "dtype_in": w["dtype_in"],
            "layout": w["layout"], "dtype_out": w["dtype_out"], "accumulate": "f32",
            "l2": "flushed between steps (read-only sweep of a 256 MB buffer)",
            "parallelism": "independent replica per GPU" if world > 1 else "1 GPU"}


PLAN_KEYS = ("block_m", "block_n", "splits", "split_tiles", "stream_k_tiles", "stages", "group_m", "grid")


def load_workload(name, dev, off):
    """Seeded host inputs of a workload and their device copies as the
    library is handed them (per the workload's layout)."""
    import torch
    import synth
    w = synth.workload(name)
    A_np = synth.matrix(w["M"], w["K"], w["dist_a"], w["seed_a"] + off, w["dtype_in"])
    B_np = synth.matrix(w["K"], w["N"], w["dist_b"], w["seed_b"] + off, w["dtype_in"])
    A_st, B_st = synth.stored(A_np, B_np, w["layout"])
    A = to_device_bits(A_st, w["dtype_in"], dev)
    B = to_device_bits(B_st, w["dtype_in"], dev)
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
    C = torch.empty((w["M"], w["N"]), dtype=tdt[w["dtype_out"]], device=dev)
    return w, A_np, B_np, A_st, B_st, A, B, C


def run_ours(args):
    import torch

    from hierarchical_gemm_gb300 import tsgemm

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    off = rank_seed_offset(rank)
    w, A_np, B_np, A_st, B_st, A, B, C = load_workload(args.workload, dev, off)
    M, N, K = w["M"], w["N"], w["K"]
    din, dout = w["dtype_in"], w["dtype_out"]
    layout = w["layout"]
    force = {k: int(v) for k, v in (kv.split("=") for kv in args.plan.split(",") if kv)}
    plan = tsgemm.Plan(M, N, K, din, dout, layout=layout, **force)
    cfg = plan.config
    flush = L2Sweep(dev)
    stream = torch.cuda.current_stream(dev)
    flops = 2.0 * M * N * K
    sampler_gpu = local if (rank == 0 or world > 1) else None

    ms_max, clocks = time_plan(plan, A, B, C, args.steps, args.warmup, dev, stream, flush, sampler_gpu, world)
    launches = args.steps
    value = aggregate_tflops(flops, ms_max, world)

    # spot check of this run's output against the oracle (sampled outputs)
    parity = sampled_parity(C, A_np, B_np, w) if rank == 0 else None

    # End to end through the C ABI with pinned host buffers.  Every step
    # uploads its A and B from pinned host memory, runs the GEMM and reads C
    # back; steps are pipelined over three streams (upload, compute,
    # download) with two device buffer sets, so one step's copies overlap
    # its neighbours' GEMMs.
    e2e = None
    if not args.no_e2e:
        e2e_steps = args.e2e_steps or min(args.steps, 50)
        A_pin = to_device_bits(A_st, din, pin=True)
        B_pin = to_device_bits(B_st, din, pin=True)
        C_pin = torch.empty((M, N), dtype=C.dtype).pin_memory()
        A_d = [torch.empty_like(A) for _ in range(2)]
        B_d = [torch.empty_like(B) for _ in range(2)]
        C_d = [torch.empty_like(C) for _ in range(2)]
        plans = [tsgemm.Plan(M, N, K, din, dout, layout=layout, **force) for _ in range(2)]
        s_up, s_gemm, s_down = (torch.cuda.Stream(dev) for _ in range(3))
        ev = lambda: torch.cuda.Event()  # noqa: E731
        up_done, gemm_done, down_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

        def e2e_step(i, first):
            j = i % 2
            with torch.cuda.stream(s_up):
                if not first[j]:
                    s_up.wait_event(gemm_done[j])       # the GEMM that read slot j is done
                A_d[j].copy_(A_pin, non_blocking=True)
                B_d[j].copy_(B_pin, non_blocking=True)
                up_done[j].record(s_up)
            s_gemm.wait_event(up_done[j])
            if not first[j]:
                s_gemm.wait_event(down_done[j])         # C of slot j has been read back
            plans[j].run(A_d[j], B_d[j], C_d[j], s_gemm)
            gemm_done[j].record(s_gemm)
            with torch.cuda.stream(s_down):
                s_down.wait_event(gemm_done[j])
                C_pin.copy_(C_d[j], non_blocking=True)
                down_done[j].record(s_down)
            first[j] = False

        first = [True, True]
        for i in range(4):
            e2e_step(i, first)
        torch.cuda.synchronize(dev)
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s_up)
        s_gemm.wait_event(e0)
        s_down.wait_event(e0)
        for i in range(e2e_steps):
            e2e_step(i, first)
        s_down.wait_stream(s_up)
        s_down.wait_stream(s_gemm)
        e1.record(s_down)
        torch.cuda.synchronize(dev)
        barrier(world)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)
        e2e = {"value": aggregate_tflops(flops, e2e_ms, world), "unit": "TFLOP/s",
               "h2d_bytes_per_step": A_pin.numel() * A_pin.element_size() + B_pin.numel() * B_pin.element_size(),
               "d2h_bytes_per_step": C_pin.numel() * C_pin.element_size(),
               "ms_per_step": e2e_ms, "steps": e2e_steps,
               "pipeline": "upload / GEMM / download streams, two device buffer sets"}
        if any(pl.status() != 0 for pl in plans):
            raise RuntimeError("device status after the end-to-end loop")
        for pl in plans:
            pl.close()
        del A_pin, B_pin, C_pin, A_d, B_d, C_d

    roofline = gemm_roofline(w, ms_max, clocks, cfg)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, rows, secs, used = oracle_rows_tflops(A_np, B_np, din, args.cpu_seconds)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": used, "kind": "oracle",
               "sample": "rows 0..%d of the %dx%dx%d product (%.1f s)" % (rows - 1, M, N, K, secs)}
    plan.close()
    del A, B, C

    # Every other benchmark configuration (and the 8-bit workloads), each
    # timed the same way over the same number of steps.
    names = EXTRA_DEFAULT if args.workloads == "all" else \
        ([] if args.workloads == "none" else [x for x in args.workloads.split(",") if x])
    workloads = {}
    for name in names:
        if name == w["name"]:
            continue
        wx, Ax_np, Bx_np, _, _, Ax, Bx, Cx = load_workload(name, dev, off)
        px = tsgemm.Plan(wx["M"], wx["N"], wx["K"], wx["dtype_in"], wx["dtype_out"], layout=wx["layout"])
        cx = px.config
        ms_x, clocks_x = time_plan(px, Ax, Bx, Cx, args.steps, args.warmup, dev, stream, flush, sampler_gpu,
                                   world)
        workloads[name] = {
            "ms_per_step": ms_x, "steps": args.steps, "gpu_launches": args.steps,
            "value": aggregate_tflops(wx["flops"], ms_x, world), "unit": "TFLOP/s",
            "config": {"M": wx["M"], "N": wx["N"], "K": wx["K"], "dtype_in": wx["dtype_in"],
                       "dtype_out": wx["dtype_out"], "layout": wx["layout"],
                       "plan": {k: cx[k] for k in PLAN_KEYS}},
            "roofline": gemm_roofline(wx, ms_x, clocks_x, cx),
            "clocks": clocks_x,
            "parity": sampled_parity(Cx, Ax_np, Bx_np, wx) if rank == 0 else None,
        }
        px.close()
        del Ax, Bx, Cx, Ax_np, Bx_np

    if rank != 0:
        return None
    return {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": din, "data": "synthetic",
        "config": gemm_config(w, world),
        "plan": {k: cfg[k] for k in PLAN_KEYS},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
        "parity": parity,
        "workloads": workloads,
    }


# ------------------------------------------------------------ attention --

ATTN_METRIC = "attention TFLOP/s (4 D flops per visible query-key pair)"


def attn_inputs(w, off=0):
    """Q, K, V bit patterns (B, H, S, D) of an attention workload, N(0, 1)."""
    import synth
    D = w["D"]

    def mk(shape, seed):
        return synth.matrix(int(np.prod(shape)) // D, D, ("normal", 1.0), seed + off, w["dtype"]).reshape(shape)
    shape_q = (w["B"], w["H"], w["Sq"], D)
    shape_k = (w["B"], w["H"], w["Sk"], D)
    return mk(shape_q, w["seed_q"]), mk(shape_k, w["seed_k"]), mk(shape_k, w["seed_v"])


def attn_sample_flops(w, rows=128):
    """Flops of attn_oracle_sample: 4 D per visible pair of the last rows."""
    Sq, Sk = w["Sq"], w["Sk"]
    i = np.arange(Sq - rows, Sq, dtype=np.int64)
    pairs = np.clip(i + Sk - Sq + 1, 0, Sk).sum() if w["causal"] else rows * Sk
    return 4.0 * w["D"] * float(pairs)


def run_attention_reference(args):
    """The oracle timed as the reference arm on an attention workload: every
    step is the last 128 query rows of one head."""
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import synth
    w = synth.attn_workload(args.workload)
    Qb, Kb, Vb = attn_inputs(w)
    for _ in range(args.warmup):
        attn_oracle_sample(w, Qb, Kb, Vb)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        attn_oracle_sample(w, Qb, Kb, Vb)
    dt = (time.perf_counter() - t0) / args.steps
    value = attn_sample_flops(w) / dt / 1e12
    return {
        "impl": "reference", "metric": ATTN_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w["name"], "B": w["B"], "H": w["H"], "Sq": w["Sq"], "Sk": w["Sk"], "D": w["D"],
                   "causal": w["causal"], "sample_rows": 128},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                         "sample": "the last 128 query rows of head (0, 0) per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def attn_oracle_sample(w, Qb, Kb, Vb, rows=128):
    """The oracle on the last `rows` query rows of head (0, 0) (the causal
    limit t <= i + Sk - Sq is unchanged when the first rows are dropped)."""
    import oracle
    q = np.ascontiguousarray(Qb[:1, :1, -rows:])
    return oracle.attention(q, Kb[:1, :1], Vb[:1, :1], w["dtype"], w["D"] ** -0.5, w["causal"])


def run_attention(args):
    import numpy as np  # noqa: F811
    import torch

    import oracle
    import synth
    from hierarchical_gemm_gb300 import tsgemm

    rank, world, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    w = synth.attn_workload(args.workload)
    Qb, Kb, Vb = attn_inputs(w, rank_seed_offset(rank))
    D, dt = w["D"], w["dtype"]
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[dt]
    to = lambda x: torch.from_numpy(x.reshape(-1).view(np.int16)).to(dev).view(tdt).reshape(x.shape)  # noqa: E731
    Q, K, V = to(Qb), to(Kb), to(Vb)
    O = torch.empty_like(Q)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = L2Sweep(dev)
    stream = torch.cuda.current_stream(dev)
    scale = D ** -0.5
    for _ in range(args.warmup):
        flush()
        tsgemm.attention(Q, K, V, scale=scale, causal=w["causal"], O=O, status=status, stream=stream)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local) if rank == 0 or world > 1 else None
    if sampler:
        sampler.start()
        time.sleep(0.25)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    for i in range(args.steps):
        flush()
        starts[i].record(stream)
        tsgemm.attention(Q, K, V, scale=scale, causal=w["causal"], O=O, status=status, stream=stream)
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    t1 = time.time()
    clocks = None
    if sampler:
        sampler.mark(t0, t1)
        clocks = sampler.stop()
    if int(status.item()) != 0:
        raise RuntimeError("attention device status %d" % int(status.item()))
    ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / args.steps
    ms_max = max_over_ranks(ms, world, dev)
    value = aggregate_tflops(w["flops"], ms_max, world)
    parity = None
    if rank == 0:
        ref, bound = attn_oracle_sample(w, Qb, Kb, Vb)
        got = O[:1, :1, -128:].cpu().reshape(-1).view(torch.int16).numpy().view(np.uint16).reshape(ref.shape)
        ok, info = oracle.accept_attention(got, ref, bound, dt)
        parity = {"sampled_outputs": int(ref.size), "ok": bool(ok),
                  "max_err_over_bound": info.get("max_err_over_bound")}
    peak, peak_desc = bf16_peak(clocks)
    achieved = w["flops"] / (ms * 1e-3) / 1e12
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        t_c = time.perf_counter()
        attn_oracle_sample(w, Qb, Kb, Vb)
        dt_c = time.perf_counter() - t_c
        cpu = {"value": attn_sample_flops(w) / dt_c / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
               "sample": "the last 128 query rows of one head (%.2f s)" % dt_c}
    if rank != 0:
        return None
    return {
        "metric": ATTN_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dt, "data": "synthetic",
        "config": {"workload": w["name"], "B": w["B"], "H": w["H"], "Sq": w["Sq"], "Sk": w["Sk"], "D": D,
                   "causal": w["causal"], "l2": "flushed between steps (read-only sweep of a 256 MB buffer)",
                   "parallelism": "independent replica per GPU" if world > 1 else "1 GPU"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": stored_traffic(w["name"]),
                     "peak_kind": peak_desc,
                     "kernel": "attn_fwd_sm103", "algorithmic_flops_per_launch": w["flops"],
                     "algorithmic_bytes_per_launch": 2 * 4 * w["B"] * w["H"] * max(w["Sq"], w["Sk"]) * w["D"]},
        "cpu_baseline": cpu, "e2e": None, "gpu_launches": args.steps, "clocks": clocks, "parity": parity,
    }


# ----------------------------------------------------------- MLA decode --

MLA_METRIC = "MLA decode HBM GB/s (Q, KV caches read once, O written once)"


def mla_oracle_sample(w, bits, batch=0, heads=32):
    """The oracle on the first `heads` heads of one batch."""
    import oracle
    q, qpe, kv, kpe = bits
    sel = (q[batch:batch + 1, :heads], qpe[batch:batch + 1, :heads], kv[batch:batch + 1], kpe[batch:batch + 1])
    return oracle.mla_decode(*sel, w["dtype"], w["scale"])


def mla_sample_bytes(w, heads=32):
    """Algorithmic bytes of the oracle sample: one batch's caches, `heads`
    heads of its queries and outputs."""
    return 2 * (w["Skv"] * (w["dim"] + w["pe_dim"]) + heads * (w["dim"] + w["pe_dim"] + w["dim"]))


def run_mla_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import synth
    w = synth.mla_workload(args.workload)
    bits = synth.mla_inputs(w)
    for _ in range(args.warmup):
        mla_oracle_sample(w, bits)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        mla_oracle_sample(w, bits)
    dt = (time.perf_counter() - t0) / args.steps
    value = mla_sample_bytes(w) / dt / 1e9
    cfg = {"workload": w["name"], "B": w["B"], "H": w["H"], "Skv": w["Skv"], "dim": w["dim"],
           "pe_dim": w["pe_dim"], "l2": "flushed between steps (read-only sweep of a 256 MB buffer)",
           "parallelism": "1 GPU"}
    return {
        "impl": "reference", "metric": MLA_METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "32 heads of batch 0 against its whole cache per step"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def run_mla(args):
    import torch

    import oracle
    import synth
    from hierarchical_gemm_gb300 import tsgemm

    rank, world, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    w = synth.mla_workload(args.workload)
    bits = synth.mla_inputs(w, rank_seed_offset(rank))
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[w["dtype"]]
    to = lambda x: torch.from_numpy(x.reshape(-1).view(np.int16)).to(dev).view(tdt).reshape(x.shape)  # noqa: E731
    q, qpe, kv, kpe = (to(x) for x in bits)
    O = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = L2Sweep(dev)
    stream = torch.cuda.current_stream(dev)
    force = {k: int(v) for k, v in (kv_.split("=") for kv_ in args.plan.split(",") if kv_)}
    pf = force.get("prefetch_blocks", 0)

    def launch():
        tsgemm.mla_decode(q, qpe, kv, kpe, scale=w["scale"], O=O, status=status, stream=stream,
                          prefetch_blocks=pf)
    for _ in range(args.warmup):
        flush()
        launch()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local) if rank == 0 or world > 1 else None
    if sampler:
        sampler.start()
        time.sleep(0.25)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    for i in range(args.steps):
        flush()
        starts[i].record(stream)
        launch()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    t1 = time.time()
    clocks = None
    if sampler:
        sampler.mark(t0, t1)
        clocks = sampler.stop()
    if int(status.item()) != 0:
        raise RuntimeError("MLA decode device status %d" % int(status.item()))
    ms = sum(s_.elapsed_time(e) for s_, e in zip(starts, ends)) / args.steps
    ms_max = max_over_ranks(ms, world, dev)
    value = world * w["bytes"] / (ms_max * 1e-3) / 1e9
    parity = None
    if rank == 0:
        ref, bound = mla_oracle_sample(w, bits)
        got = O[:1, :32].cpu().reshape(-1).view(torch.int16).numpy().view(np.uint16).reshape(ref.shape)
        ok, info = oracle.accept_attention(got, ref, bound, w["dtype"])
        parity = {"sampled_outputs": int(ref.size), "ok": bool(ok),
                  "max_err_over_bound": info.get("max_err_over_bound")}
    peaks, kind = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    tensor_peak, tensor_desc = bf16_peak(clocks)
    achieved = w["bytes"] / (ms * 1e-3) / 1e9
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        t_c = time.perf_counter()
        mla_oracle_sample(w, bits)
        dt_c = time.perf_counter() - t_c
        cpu = {"value": mla_sample_bytes(w) / dt_c / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": "32 heads of batch 0 against its whole cache (%.2f s)" % dt_c}
    if rank != 0:
        return None
    return {
        "metric": MLA_METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w["dtype"], "data": "synthetic",
        "config": {"workload": w["name"], "B": w["B"], "H": w["H"], "Skv": w["Skv"], "dim": w["dim"],
                   "pe_dim": w["pe_dim"], "l2": "flushed between steps (read-only sweep of a 256 MB buffer)",
                   "parallelism": "independent replica per GPU" if world > 1 else "1 GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": stored_traffic(w["name"]), "peak_kind": kind + " HBM copy bandwidth",
                     "kernel": "mla_decode_sm103", "algorithmic_bytes_per_launch": w["bytes"],
                     "algorithmic_flops_per_launch": w["flops"],
                     "tensor_tflops": w["flops"] / (ms * 1e-3) / 1e12, "tensor_peak": tensor_peak,
                     "tensor_peak_kind": tensor_desc},
        "cpu_baseline": cpu, "e2e": None, "gpu_launches": args.steps, "clocks": clocks, "parity": parity,
    }


def main(argv=None):
    args = parse_args(argv)
    if args.workload.startswith("mla_"):
        out = run_mla_reference(args) if args.impl == "reference" else run_mla(args)
    elif args.workload.startswith("attn_"):
        out = run_attention_reference(args) if args.impl == "reference" else run_attention(args)
    else:
        out = run_reference(args) if args.impl == "reference" else run_ours(args)
    if out is not None:
        print(json.dumps(out), flush=True)
    rank, world, _ = dist_env()
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
