"""Benchmark: quant-matvec weight GB/s on GB300 for one decode token.

Default workload (one "step"): every projection matvec of one decode token of
an 8B-dense-shaped model in Q8_0, n_vec = 1 -- 32 layers x (q 4096x4096,
k 1024x4096, v 1024x4096, o 4096x4096, gate 14336x4096, up 14336x4096,
down 4096x14336) plus the lm_head 128256x4096: 225 matvecs, 7,973,699,584
weight bytes, all distinct (7.97 GB > L2, so no flush is needed).  Weights are
seeded synthetic N(0, 0.02) fp32, quantized on the GPU; each matvec gets its
own x ~ N(0, 1).  The step is captured once as a CUDA graph and replayed.

value      = weight bytes per step / device time per step (GB/s, 1e9 B),
             summed over ranks (replicas, weak scaling).
e2e        = the same, with each step's x copied host->device from pinned
             memory and every y copied back inside the timed region.
roofline   = the matvec kernel's algorithmic bytes (weights + x + y) per
             launch / its mean launch time, from CUDA event pairs around every
             launch of the step (a second captured graph), against the
             measured HBM copy bandwidth.
cpu_baseline = the CPU oracle (plain C, one thread) on a bounded sample of the
             same matrices.

--impl reference times that oracle as the reference arm (on the host cores).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from quantized_weight_matvec_hq_gb300 import synthetic  # noqa: E402

# name -> (model shape, format, q|k|v and gate|up row-fused)
WORKLOADS = {
    "8b-q8_0": ("8b-dense", "q8_0", True),
    "8b-q8_0-unfused": ("8b-dense", "q8_0", False),
    "8b-q4_0": ("8b-dense", "q4_0", True),
    "8b-q4_0-unfused": ("8b-dense", "q4_0", False),
    "qwen3-0.6b-q8_0": ("qwen3-0.6b", "q8_0", True),
    "qwen3-0.6b-q8_0-unfused": ("qwen3-0.6b", "q8_0", False),
}


def workload_matrices(name, shape=None, fmt=None):
    """(model, format, [(name, rows, cols), ...]) of one step.  With `shape`
    ("ROWSxCOLS"), the step is enough distinct copies of that one matrix to
    exceed 4x the L2 (>= 520 MB) so that no launch reads from L2."""
    if shape:
        rows, cols = (int(v) for v in shape.lower().split("x"))
        one = weight_bytes(fmt, rows, cols)
        copies = max(4, -(-520_000_000 // one))
        return f"single {rows}x{cols}", fmt, [(f"m{rows}x{cols}", rows, cols)] * copies
    model, fmt, fused = WORKLOADS[name]
    return model, fmt, synthetic.decode_token_shapes(model, fused)


def weight_bytes(fmt, rows, cols):
    return rows * (cols // 32) * (34 if fmt == "q8_0" else 18)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        try:
            lines = open(self.path).read().strip().splitlines()
        except OSError:
            lines = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if self.path:
            os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    """(world size, rank, local rank) from the torchrun environment."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(values, device):
    """Element-wise max of per-rank timings (the slowest replica sets the step
    time); needs an initialised process group."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def aggregate_value(world, bytes_per_step, ms_per_step):
    """Whole-job weight GB/s: every replica streams bytes_per_step per step."""
    return world * bytes_per_step / (ms_per_step / 1e3) / 1e9


def read_traffic(path, workload, n_vec, shape):
    """DRAM bytes (read + write) per step of the matvec kernel, from a line
    `<workload> n_vec=<k> dram_bytes_per_step=<int>` of the ncu summary file;
    None when the file has no line for this configuration."""
    if shape or not os.path.exists(path):
        return None
    for ln in open(path):
        parts = ln.split()
        if len(parts) >= 3 and parts[0] == workload and parts[1] == f"n_vec={n_vec}" \
                and parts[2].startswith("dram_bytes_per_step="):
            return int(parts[2].split("=", 1)[1])
    return None


# ----------------------------------------------------------------- CUDA helpers

def _cudart():
    import torch  # noqa: F401  (loads torch's runtime first)
    for name in ("libcudart.so.13", "libcudart.so.12", "libcudart.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    for p in ("/usr/local/cuda/lib64/libcudart.so.13", "/usr/local/cuda/lib64/libcudart.so"):
        if os.path.exists(p):
            return ctypes.CDLL(p)
    raise OSError("libcudart not found")


class Step:
    """One decode token's matvecs, resident in HBM, launched through the C ABI."""

    def __init__(self, name, n_vec, device, seed, shape=None, fmt=None):
        import torch
        import quantized_weight_matvec_hq_gb300 as hq
        self.hq = hq
        self.torch = torch
        self.model, self.fmt, self.shapes = workload_matrices(name, shape, fmt)
        self.n_vec = n_vec
        self.device = device
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        total = sum(weight_bytes(self.fmt, r, c) for (_, r, c) in self.shapes)
        free, _ = torch.cuda.mem_get_info(device)
        if total > 0.8 * free:
            raise RuntimeError(f"workload needs {total / 1e9:.1f} GB, only {free / 1e9:.1f} GB free")
        self.W, self.x, self.y = [], [], []
        quant = hq.hq_quantize_q8_0 if self.fmt == "q8_0" else hq.hq_quantize_q4_0
        # every matvec's x and y live in one contiguous buffer each (16-byte
        # aligned views), so a step's inputs and outputs cross PCIe/C2C in one copy
        xo, yo = [], []
        nx = ny = 0
        for (_, rows, cols) in self.shapes:
            xo.append(nx)
            yo.append(ny)
            nx += -(-n_vec * cols // 4) * 4
            ny += -(-n_vec * rows // 4) * 4
        self.x_all = torch.randn(nx, generator=g, device=device, dtype=torch.float32)
        self.y_all = torch.empty(ny, device=device, dtype=torch.float32)
        for i, (_, rows, cols) in enumerate(self.shapes):
            wf = torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32).mul_(0.02)
            wq = torch.empty((rows, weight_bytes(self.fmt, 1, cols)), dtype=torch.uint8, device=device)
            quant(wf, wq, rows, cols)
            del wf
            self.W.append(wq)
            self.x.append(self.x_all[xo[i]:xo[i] + n_vec * cols].view(n_vec, cols))
            self.y.append(self.y_all[yo[i]:yo[i] + n_vec * rows].view(n_vec, rows))
        torch.cuda.synchronize()
        self.fn = hq.hq_matvec_q8_0 if self.fmt == "q8_0" else hq.hq_matvec_q4_0
        self.weight_bytes = sum(weight_bytes(self.fmt, r, c) for (_, r, c) in self.shapes)
        self.x_bytes = int(self.x_all.numel()) * 4
        self.y_bytes = int(self.y_all.numel()) * 4

    def launch_all(self, stream, events=None):
        for i, (_, rows, cols) in enumerate(self.shapes):
            if events is not None:
                events.record_before(i, stream)
            self.fn(self.W[i], self.x[i], self.y[i], rows, cols, self.n_vec, stream=stream)
            if events is not None:
                events.record_after(i, stream)

    def capture(self, events=None):
        torch = self.torch
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):               # warm the path (attribute set-up) before capture
            self.launch_all(s.cuda_stream)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            self.launch_all(torch.cuda.current_stream().cuda_stream, events)
        torch.cuda.synchronize()
        return graph


class LaunchEvents:
    """Event pairs around every launch, recorded as external event nodes of a
    captured graph so their times are readable after each replay."""

    def __init__(self, n, cudart):
        self.rt = cudart
        self.rt.cudaEventCreate.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
        self.rt.cudaEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
        self.rt.cudaEventElapsedTime.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_void_p, ctypes.c_void_p]
        self.rt.cudaEventSynchronize.argtypes = [ctypes.c_void_p]
        self.before = [self._new() for _ in range(n)]
        self.after = [self._new() for _ in range(n)]

    def _new(self):
        e = ctypes.c_void_p()
        rc = self.rt.cudaEventCreate(ctypes.byref(e))
        if rc != 0:
            raise RuntimeError(f"cudaEventCreate failed ({rc})")
        return e

    def record_before(self, i, stream):
        rc = self.rt.cudaEventRecordWithFlags(self.before[i], ctypes.c_void_p(stream), 1)  # external
        if rc != 0:
            raise RuntimeError(f"cudaEventRecordWithFlags failed ({rc})")

    def record_after(self, i, stream):
        rc = self.rt.cudaEventRecordWithFlags(self.after[i], ctypes.c_void_p(stream), 1)
        if rc != 0:
            raise RuntimeError(f"cudaEventRecordWithFlags failed ({rc})")

    def durations_ms(self):
        self.rt.cudaEventSynchronize(self.after[-1])
        out = []
        for b, a in zip(self.before, self.after):
            t = ctypes.c_float()
            rc = self.rt.cudaEventElapsedTime(ctypes.byref(t), b, a)
            if rc != 0:
                raise RuntimeError(f"cudaEventElapsedTime failed ({rc})")
            out.append(t.value)
        return out


# ----------------------------------------------------------------- CPU oracle timing

class OracleSample:
    """The C oracle (one thread) on a bounded sample of the workload: the first
    rows (about 4M weights) of each distinct matrix shape of the token,
    quantized by the oracle itself.  One pass = one matvec per shape."""

    def __init__(self, name, n_vec, seed=synthetic.SEED_BASE + 2):
        import oracle
        self.oracle = oracle
        self.model, self.fmt, shapes = workload_matrices(name)
        self.n_vec = n_vec
        distinct = []
        for s_ in shapes:
            if (s_[1], s_[2]) not in [(d[1], d[2]) for d in distinct]:
                distinct.append(s_)
        g = synthetic.rng(seed)
        self.slabs = []
        for (nm, rows, cols) in distinct:
            r = min(rows, max(8, (1 << 22) // cols))
            W = synthetic.weights(g, r, cols)
            blocks = oracle.quantize_q8_0(W) if self.fmt == "q8_0" else oracle.quantize_q4_0(W)
            self.slabs.append((nm, r, cols, blocks, synthetic.activations(g, n_vec, cols)))
        self.pass_bytes = sum(weight_bytes(self.fmt, r, c) for (_, r, c, _, _) in self.slabs)

    def run_pass(self):
        for (_, r, cols, blocks, x) in self.slabs:
            self.oracle.matvec(self.fmt, blocks, x, r, cols)
        return self.pass_bytes

    def describe(self, passes):
        return (f"{passes} passes; each = the first rows (~4M weights) of each of the {len(self.slabs)} "
                f"distinct {self.model} matrix shapes, {self.pass_bytes / 1e6:.1f} MB of {self.fmt}, "
                f"n_vec={self.n_vec}, single-threaded C oracle with f64 accumulation")

    def timed(self, budget_s):
        done, n, t0 = 0, 0, time.perf_counter()
        while True:
            done += self.run_pass()
            n += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                return done / el / 1e9, self.describe(n), el


# ----------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["hq", "reference"], default="hq")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="8b-q8_0")
    ap.add_argument("--n-vec", type=int, default=1)
    ap.add_argument("--shape", default=None,
                    help="time one matrix shape ROWSxCOLS instead of a decode token (profiling aid)")
    ap.add_argument("--format", choices=["q8_0", "q4_0"], default="q8_0", help="format for --shape")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--traffic-file", default=os.path.join(ROOT, "profiles", "dram_traffic.txt"),
                    help="DRAM bytes per step of the matvec kernel, from an ncu capture (text)")
    args = ap.parse_args()

    world, rank, local_rank = dist_env()
    model, fmt, shapes = workload_matrices(args.workload, args.shape, args.format)
    fused_note = (" with q|k|v and gate|up row-fused (same input)" if WORKLOADS[args.workload][2]
                  else ", every projection its own call")
    config = {"workload": (f"{model} decode token, {fmt}, n_vec={args.n_vec}: "
                           f"{len(shapes)} matvecs (all projections + lm_head){fused_note}") if not args.shape else
                          (f"{len(shapes)} distinct {args.shape} {fmt} matrices per step, n_vec={args.n_vec}"),
              "model_shape": model, "format": fmt, "n_vec": args.n_vec, "matvecs_per_step": len(shapes),
              "l2": "inputs larger than L2 (all weights distinct, 7.97 GB Q8_0 / 4.2 GB Q4_0 per step)"
              if model == "8b-dense" else "all weights distinct per step",
              "seed": synthetic.SEED_BASE + 2}

    if args.impl == "reference":
        if world > 1 and rank != 0:
            return
        samp = OracleSample(args.workload, args.n_vec)
        for _ in range(args.warmup):
            samp.run_pass()
        times = []
        for _ in range(args.steps):
            t0 = time.perf_counter()
            samp.run_pass()
            times.append(time.perf_counter() - t0)
        value = samp.pass_bytes * len(times) / sum(times) / 1e9
        line = {"impl": "reference", "metric": "quant-matvec weight GB/s", "value": round(value, 4),
                "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(1e3 * sum(times) / len(times), 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": config,
                "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                                 "sample": samp.describe(args.steps) + " (one pass per step)"},
                "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)

    step = Step(args.workload, args.n_vec, device, synthetic.SEED_BASE + 2 + rank, args.shape, args.format)
    graph = step.capture()
    events = LaunchEvents(len(shapes), _cudart())
    graph_ev = step.capture(events)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    # ---- device-resident timing
    for _ in range(args.warmup):
        graph.replay()
    barrier()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        start.record()
        for _ in range(args.steps):
            graph.replay()
        end.record()
        end.synchronize()
        dev_ms = start.elapsed_time(end) / args.steps
        # ---- per-launch durations (event pairs around each launch), same steps
        per_launch = np.zeros(len(shapes))
        for _ in range(args.steps):
            graph_ev.replay()
            per_launch += np.array(events.durations_ms())
        per_launch /= args.steps
        # ---- end to end: pinned host x in, y out, every step
        x_host = step.x_all.cpu().pin_memory()
        y_host = torch.empty(step.y_all.shape, dtype=torch.float32).pin_memory()
        for _ in range(2):
            step.x_all.copy_(x_host, non_blocking=True)
            graph.replay()
            y_host.copy_(step.y_all, non_blocking=True)
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            step.x_all.copy_(x_host, non_blocking=True)
            graph.replay()
            y_host.copy_(step.y_all, non_blocking=True)
        e1.record()
        e1.synchronize()
        e2e_ms = e0.elapsed_time(e1) / args.steps
    clk = clocks.summary()

    if world > 1:
        dev_ms, e2e_ms = max_over_ranks([dev_ms, e2e_ms], device)

    if rank != 0:
        torch.distributed.destroy_process_group()
        return

    peak, peak_kind = load_peaks()
    value = aggregate_value(world, step.weight_bytes, dev_ms)
    e2e = aggregate_value(world, step.weight_bytes, e2e_ms)
    # Roofline of the matvec kernel: the step consists of its launches only, so
    # the mean launch duration is the step's device time over the launch count.
    # The event pairs of the per-shape breakdown add a few microseconds per
    # launch and break the programmatic-launch overlap: a breakdown only.
    alg = np.array([weight_bytes(fmt, r, c) + 4 * args.n_vec * (r + c) for (_, r, c) in shapes], dtype=np.float64)
    achieved = float(alg.sum() / (dev_ms / 1e3) / 1e9)
    traffic = read_traffic(args.traffic_file, args.workload, args.n_vec, args.shape)
    kernel_ms = float(per_launch.sum())
    by_shape = {}
    for (nm, r, c), ms, b in zip(shapes, per_launch, alg):
        k = f"{nm} {r}x{c}"
        d = by_shape.setdefault(k, [0.0, 0.0, 0])
        d[0] += ms
        d[1] += b
        d[2] += 1
    shapes_out = {k: {"launches": v[2], "us_per_launch": round(v[0] / v[2] * 1e3, 3),
                      "gbs": round(v[1] / (v[0] / 1e3) / 1e9, 1)}
                  for k, v in by_shape.items()}

    line = {
        "metric": "quant-matvec weight GB/s", "value": round(value, 2), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dev_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp32 accumulate over " + fmt, "data": "synthetic", "config": config,
        "tok_per_s": round(1e3 / dev_ms * world, 2),
        "frac_of_hbm": round(value / world / peak, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": (round(traffic / len(shapes)) if traffic is not None else None),
                     "traffic_unit": "DRAM bytes read+written per launch (mean over the step), from ncu",
                     "algorithmic_bytes_per_launch": round(float(alg.sum()) / len(shapes)),
                     "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs), burst",
                     "kernel": "matvec_tma_kernel (every launch of the step)",
                     "launches_per_step": len(shapes),
                     "mean_launch_us": round(dev_ms * 1e3 / len(shapes), 3)},
        "per_shape_event_pairs": shapes_out,
        "per_shape_event_pairs_ms_per_step": round(kernel_ms, 4),
        "e2e": {"value": round(e2e, 2), "unit": "GB/s", "ms_per_step": round(e2e_ms, 5),
                "h2d_bytes_per_step": int(step.x_bytes), "d2h_bytes_per_step": int(step.y_bytes)},
        "gpu_launches": len(shapes) * args.steps,
        "clocks": clk,
    }
    if not args.no_cpu_baseline and not args.shape:
        gbs, desc, el = OracleSample(args.workload, args.n_vec).timed(args.cpu_budget)
        line["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "sample": desc, "seconds": round(el, 2)}
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
