#!/usr/bin/env python
"""Benchmark of the tile-level GEMM C = A * B on GB300.

One step is one C = A * B of the benchmark workload (default: M = N = K =
4096, bf16 inputs drawn from N(0, 1), fp32 accumulation, bf16 output) on
inputs already resident in HBM.  The L2 cache (129 MB, larger than the
96 MB working set) is flushed between steps by writing a 256 MB buffer; each
step's GEMM is timed with CUDA events on the launching stream.

Prints one JSON line.  `value` is TFLOP/s (2*M*N*K per step) over all ranks;
`e2e` is the same metric through the same C ABI call with pinned host
buffers, the host->device copies of A and B and the device->host copy of C
inside the timed region; `roofline` relates the kernel to the measured bf16
tensor peak (for 8-bit inputs: twice that, the nominal fp8 : bf16 ratio);
`cpu_baseline` is the fp64 oracle timed on the host cores.  --workload picks
another seeded workload (the five benchmark configurations, or the FP8 ones).

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

# Source files whose change invalidates a stored ncu traffic figure.
KERNEL_SOURCES = ["hierarchical_gemm_gb300/csrc/gemm_sm103.cuh",
                  "hierarchical_gemm_gb300/csrc/gemm_sm103_2sm.cuh",
                  "hierarchical_gemm_gb300/csrc/ptx.cuh",
                  "hierarchical_gemm_gb300/csrc/kernels_1sm.cu",
                  "hierarchical_gemm_gb300/csrc/kernels_2sm.cu"]
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
                    help="force plan fields, e.g. block_m=256,block_n=128,splits=1")
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


ATTN_SOURCES = ["hierarchical_gemm_gb300/csrc/attention_sm103.cu",
                "hierarchical_gemm_gb300/csrc/ptx.cuh"]


def kernel_source_hash(sources=None):
    h = hashlib.sha256()
    for rel in sources or KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def stored_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    with the current kernel source (the files the entry names); else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(workload)
    if not e or e.get("source_hash") != kernel_source_hash(e.get("sources")):
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
        "config": {"workload": w["name"], "M": w["M"], "N": w["N"], "K": w["K"],
                   "dtype_in": w["dtype_in"], "dtype_out": w["dtype_out"],
                   "sample_rows": rows},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": used, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


# ------------------------------------------------------------------ ours --

def run_ours(args):
    import numpy as np
    import torch

    import synth
    from hierarchical_gemm_gb300 import tsgemm

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    w = synth.workload(args.workload)
    M, N, K = w["M"], w["N"], w["K"]
    din, dout = w["dtype_in"], w["dtype_out"]
    layout = w["layout"]
    off = rank_seed_offset(rank)
    A_np = synth.matrix(M, K, w["dist_a"], w["seed_a"] + off, din)
    B_np = synth.matrix(K, N, w["dist_b"], w["seed_b"] + off, din)
    A_st, B_st = synth.stored(A_np, B_np, layout)  # as the library is handed them
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
    A = to_device_bits(A_st, din, dev)
    B = to_device_bits(B_st, din, dev)
    C = torch.empty((M, N), dtype=tdt[dout], device=dev)
    force = {k: int(v) for k, v in (kv.split("=") for kv in args.plan.split(",") if kv)}
    plan = tsgemm.Plan(M, N, K, din, dout, layout=layout, **force)
    cfg = plan.config
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    flops = 2.0 * M * N * K

    for _ in range(args.warmup):
        flush.zero_()
        plan.run(A, B, C, stream)
    torch.cuda.synchronize(dev)
    if plan.status() != 0:
        raise RuntimeError("device status %d after warm-up" % plan.status())

    sampler = ClockSampler(local) if rank == 0 or world > 1 else None
    if sampler:
        sampler.start()
        time.sleep(0.25)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        plan.run(A, B, C, stream)
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    t_wall1 = time.time()
    launches = args.steps
    if sampler:
        sampler.mark(t_wall0, t_wall1)
        clocks = sampler.stop()
    else:
        clocks = None
    st = plan.status()
    if st != 0:
        raise RuntimeError("device status %d (%s)" % (st, tsgemm.status_string(st)))
    times = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = sum(times) / len(times)
    ms_max = max_over_ranks(ms, world, dev)
    value = aggregate_tflops(flops, ms_max, world)

    # spot check of this run's output against the oracle (sampled outputs)
    parity = None
    if rank == 0:
        import oracle
        r = np.random.default_rng(7)
        rows = r.integers(0, M, 1024)
        cols = r.integers(0, N, 1024)
        Ch = C.cpu()
        Ch = Ch.numpy() if dout == "f32" else Ch.view(torch.int16).numpy().view(np.uint16)
        ref, sabs = oracle.gemm_sampled(A_np, B_np, din, rows, cols)
        ok, info = oracle.accept(Ch[rows, cols], ref, sabs, dout)
        parity = {"sampled_outputs": int(rows.size), "ok": bool(ok),
                  "max_err_over_bound": info.get("max_err_over_bound")}

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
        C_pin = torch.empty((M, N), dtype=tdt[dout]).pin_memory()
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

    peak, peak_desc = bf16_peak(clocks)
    eight_bit = din in ("e4m3", "e5m2")
    if eight_bit:
        peak *= FP8_TO_BF16
        peak_desc += " x %.0f (nominal fp8 : bf16 dense ratio)" % FP8_TO_BF16
    algo_bytes = synth.workloads.in_nbytes(din) * (M * K + K * N) + synth.workloads.out_nbytes(dout) * M * N
    bound, achieved, peak, unit, peak_desc = roofline_point(flops, algo_bytes, ms, peak, peak_desc)
    roofline = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "traffic": stored_traffic(w["name"]),
                "peak_kind": peak_desc,
                "kernel": "gemm_sm103_%s<BN=%d%s>" % ("2sm" if cfg["block_m"] == 256 else "1sm", cfg["block_n"],
                                                     ", 8-bit" if eight_bit else ""),
                "algorithmic_flops_per_launch": flops,
                "algorithmic_bytes_per_launch": algo_bytes}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, rows, secs, used = oracle_rows_tflops(A_np, B_np, din, args.cpu_seconds)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": used, "kind": "oracle",
               "sample": "rows 0..%d of the %dx%dx%d product (%.1f s)" % (rows - 1, M, N, K, secs)}

    if rank != 0:
        return None
    return {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": din, "data": "synthetic",
        "config": {"workload": w["name"], "M": M, "N": N, "K": K, "dtype_in": din, "layout": layout,
                   "dtype_out": dout, "accumulate": "f32", "l2": "flushed between steps (256 MB write)",
                   "plan": {k: cfg[k] for k in ("block_m", "block_n", "splits", "stages", "group_m", "grid")},
                   "parallelism": "independent replica per GPU" if world > 1 else "1 GPU"},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
        "parity": parity,
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
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    scale = D ** -0.5
    for _ in range(args.warmup):
        flush.zero_()
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
        flush.zero_()
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
                   "causal": w["causal"], "l2": "flushed between steps (256 MB write)",
                   "parallelism": "independent replica per GPU" if world > 1 else "1 GPU"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": stored_traffic(w["name"]),
                     "peak_kind": peak_desc,
                     "kernel": "attn_fwd_sm103", "algorithmic_flops_per_launch": w["flops"],
                     "algorithmic_bytes_per_launch": 2 * 4 * w["B"] * w["H"] * max(w["Sq"], w["Sk"]) * w["D"]},
        "cpu_baseline": cpu, "e2e": None, "gpu_launches": args.steps, "clocks": clocks, "parity": parity,
    }


def main(argv=None):
    args = parse_args(argv)
    if args.workload.startswith("attn_"):
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
