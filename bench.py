"""Benchmark: quant-matvec weight GB/s on GB300 for one decode token.

Default workload (one "step"): every projection matvec of one decode token of
an 8B-dense-shaped model in Q8_0, n_vec = 1 -- 32 layers x (q 4096x4096,
k 1024x4096, v 1024x4096, o 4096x4096, gate 14336x4096, up 14336x4096,
down 4096x14336) plus the lm_head 128256x4096: 225 matvecs, 7,973,699,584
weight bytes, all distinct (7.97 GB > L2, so no flush is needed).  Weights are
seeded synthetic N(0, 0.02) fp32, quantized on the GPU; each matvec gets its
own x ~ N(0, 1).  The step is captured once as a CUDA graph and replayed.

Other workloads (--workload): the same token unfused, in Q4_0, or Qwen3-0.6B-
shaped; "moe-q8_0" -- 48 MoE layers, each an expert-indexed gate|up and down
launch over its own bank of 128 experts (8 active per token, drawn per layer);
"int8-requant" -- 96 distinct copies of each of the 1024x3072 and 3072x1024
int8 matrices with per-row requant.  --n-vec sets the activation vectors per
launch (1..8); for MoE the weight bytes count the distinct experts read.

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

# name -> (kind, model shape, format, q|k|v and gate|up row-fused)
WORKLOADS = {
    "8b-q8_0": ("dense", "8b-dense", "q8_0", True),
    "8b-q8_0-unfused": ("dense", "8b-dense", "q8_0", False),
    "8b-q4_0": ("dense", "8b-dense", "q4_0", True),
    "8b-q4_0-unfused": ("dense", "8b-dense", "q4_0", False),
    "8b-q4_k": ("dense", "8b-dense", "q4_k", True),
    "qwen3-0.6b-q8_0": ("dense", "qwen3-0.6b", "q8_0", True),
    "qwen3-0.6b-q8_0-unfused": ("dense", "qwen3-0.6b", "q8_0", False),
    "moe-q8_0": ("moe", "moe-128x8-hidden2048", "q8_0", True),
    "moe-q8_0-ffn": ("moe", "moe-128x8-hidden2048", "q8_0", True),
    "int8-requant": ("int8", "int8-1024x3072+3072x1024", "i8", False),
    "8b-q8_0-lora": ("dense", "8b-dense", "q8_0", True),
    "8b-q4_0-lora": ("dense", "8b-dense", "q4_0", True),
}
# QLoRA workloads: a bf16 adapter of this rank on every projection (not the
# lm_head), scale alpha / r = 2 (rank-16 adapters on the attention and FFN
# projections are the pages' example configuration)
LORA_RANK = {"8b-q8_0-lora": 16, "8b-q4_0-lora": 16}
LORA_SCALE = 2.0
# MoE feed-forward workloads: gate|up with the SwiGLU epilogue (interleaved
# gate/up rows), down with the router-weighted sum over the slots
MOE_FFN = {"moe-q8_0-ffn"}
# MoE decode: a stack of this many layers, each with its own bank of experts
# (128 x (gate|up 1536x2048 + down 2048x768) Q8_0 = 642 MB per layer)
MOE_LAYERS = 48
# int8 GEMV: this many distinct copies of each of the two matrices per step (604 MB)
INT8_COPIES = 96


class Op:
    """One launch of a step: a dense matvec, an expert-indexed MoE matvec or an
    int8 requant GEMV, with the bytes it reads and writes."""

    def __init__(self, kind, name, rows, cols, fmt, n_experts=0, n_active=0, x_per_slot=0, ids=None, label=None,
                 lora_rank=0, epi=None):
        self.kind, self.name, self.rows, self.cols, self.fmt = kind, name, rows, cols, fmt
        self.epi = epi                               # MoE epilogue: None, "swiglu" or "combine"
        self.label = label or name                   # the matrix's role, without layer or copy index
        self.lora_rank = lora_rank                   # QLoRA adapter rank (0: none)
        self.n_experts, self.n_active, self.x_per_slot, self.ids = n_experts, n_active, x_per_slot, ids

    def x_elems(self, n_vec):
        return n_vec * (self.n_active if self.x_per_slot else 1) * self.cols

    def y_elems(self, n_vec):
        if self.epi == "swiglu":
            return n_vec * self.n_active * self.rows // 2     # h = silu(gate) * up
        if self.epi == "combine":
            return n_vec * self.rows                         # the weighted sum over the slots
        return n_vec * (self.n_active if self.kind == "moe" else 1) * self.rows

    def weight_bytes(self):
        """Weight bytes one launch reads: for MoE, the distinct experts of the routing."""
        if self.kind == "int8":
            return self.rows * self.cols + 8 * self.rows               # + mult, shift
        one = weight_bytes(self.fmt, self.rows, self.cols)
        if self.kind == "moe":
            return one * len(np.unique(self.ids))
        return one + 2 * self.lora_rank * (self.rows + self.cols)     # + bf16 adapter factors

    def alg_bytes(self, n_vec):
        """Algorithmic bytes of a launch: weights read + x read + y written (+ expert ids)."""
        el = 1 if self.kind == "int8" else 4
        extra = self.ids.size * 4 if self.kind == "moe" else 0
        extra += 2 * 4 * self.lora_rank * n_vec                     # u = A x written, then read
        if self.epi == "combine":
            extra += 4 * self.ids.size                              # router weights
        return self.weight_bytes() + el * (self.x_elems(n_vec) + self.y_elems(n_vec)) + extra


def workload_ops(name, n_vec, shape=None, fmt=None, seed=synthetic.SEED_BASE + 2):
    """(model, format, [Op, ...]) of one step.  With `shape` ("ROWSxCOLS"), the
    step is enough distinct copies of that one matrix to exceed 4x the L2
    (>= 520 MB) so that no launch reads from L2."""
    if shape:
        rows, cols = (int(v) for v in shape.lower().split("x"))
        one = weight_bytes(fmt, rows, cols)
        copies = max(4, -(-520_000_000 // one))
        return f"single {rows}x{cols}", fmt, [Op("dense", f"m{rows}x{cols}", rows, cols, fmt)] * copies
    kind, model, fmt, fused = WORKLOADS[name]
    if kind == "dense":
        rank = LORA_RANK.get(name, 0)
        return model, fmt, [Op("dense", n, r, c, fmt, lora_rank=(rank if n != "lm_head" else 0))
                            for (n, r, c) in synthetic.decode_token_shapes(model, fused)]
    if kind == "moe":
        g = synthetic.rng(seed + 7)
        ops = []
        E, A, H, F = synthetic.MOE_N_EXPERTS, synthetic.MOE_N_ACTIVE, synthetic.MOE_HIDDEN, synthetic.MOE_FFN
        ffn = name in MOE_FFN
        for layer in range(MOE_LAYERS):
            ids = synthetic.expert_ids(g, n_vec, A, E)
            ops.append(Op("moe", f"gate_up{layer}", 2 * F, H, fmt, E, A, 0, ids, label="gate_up",
                          epi="swiglu" if ffn else None))
            ops.append(Op("moe", f"down{layer}", H, F, fmt, E, A, 1, ids, label="down",
                          epi="combine" if ffn else None))
        return model, fmt, ops
    ops = []
    for i in range(INT8_COPIES):
        for (r, c) in synthetic.INT8_SHAPES:
            ops.append(Op("int8", f"i8_{r}x{c}_{i}", r, c, fmt, label="i8"))
    return model, fmt, ops


def weight_bytes(fmt, rows, cols):
    if fmt == "i8":
        return rows * cols
    if fmt == "q4_k":
        return rows * (cols // 256) * 144
    return rows * (cols // 32) * (34 if fmt == "q8_0" else 18)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def read_probe_gbs(device, gib=2, reps=5):
    """A read-only HBM reference: a torch sum over a 2 GiB fp32 buffer (far
    above L2), timed with CUDA events.  Not part of the product path."""
    import torch
    buf = torch.ones(gib << 28, dtype=torch.float32, device=device)
    buf.sum()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        buf.sum()
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / reps
    n = buf.numel() * 4
    del buf
    return n / (ms / 1e3) / 1e9


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the oracle baseline line."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def fp32_flops(ops, n_vec):
    """FP32 multiply-add flops of a step: 2 per weight per vector (MoE: per chosen
    (token, slot) pair); None for the int8 path, which is not fp32 arithmetic."""
    total = 0
    for op in ops:
        if op.kind == "int8":
            return None
        pairs = n_vec * op.n_active if op.kind == "moe" else n_vec
        total += 2 * op.rows * op.cols * pairs
    return total


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
    """One step's launches, resident in HBM, launched through the C ABI.  Every
    launch's x (and, for MoE, the expert ids) and y live in one contiguous
    buffer each (16-byte aligned views), so a step's inputs and outputs cross
    the host link in one copy each."""

    def __init__(self, name, n_vec, device, seed, shape=None, fmt=None):
        import torch
        import quantized_weight_matvec_hq_gb300 as hq
        self.hq = hq
        self.torch = torch
        self.model, self.fmt, self.ops = workload_ops(name, n_vec, shape, fmt)
        self.n_vec = n_vec
        self.device = device
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        total = sum(self._stored_bytes(op) for op in self.ops)
        free, _ = torch.cuda.mem_get_info(device)
        if total > 0.8 * free:
            raise RuntimeError(f"workload needs {total / 1e9:.1f} GB, only {free / 1e9:.1f} GB free")
        xdt = torch.int8 if self.fmt == "i8" else torch.float32
        xo, yo, io = [], [], []
        nx = ny = ni = 0
        for op in self.ops:
            xo.append(nx)
            yo.append(ny)
            io.append(ni)
            nx += -(-op.x_elems(n_vec) // 16) * 16
            ny += -(-op.y_elems(n_vec) // 16) * 16
            ni += -(-(op.ids.size if op.kind == "moe" else 0) // 4) * 4
        if self.fmt == "i8":
            self.x_all = torch.randint(-127, 128, (nx,), generator=g, device=device, dtype=torch.int8)
        else:
            self.x_all = torch.randn(nx, generator=g, device=device, dtype=torch.float32)
        self.y_all = torch.empty(ny, device=device, dtype=xdt)
        self.ids_all = torch.zeros(max(ni, 4), device=device, dtype=torch.int32)
        self.W, self.x, self.y, self.ids, self.mult, self.shift = [], [], [], [], [], []
        self.lora = []                              # (A, B, workspace) per op, or None
        self.comb = []                              # router weights per op, or None
        for i, op in enumerate(self.ops):
            self.x.append(self.x_all[xo[i]:xo[i] + op.x_elems(n_vec)])
            self.y.append(self.y_all[yo[i]:yo[i] + op.y_elems(n_vec)])
            if op.kind == "moe":
                v = self.ids_all[io[i]:io[i] + op.ids.size]
                v.copy_(torch.from_numpy(op.ids.reshape(-1)))
                self.ids.append(v)
            else:
                self.ids.append(None)
            self.W.append(self._weights(op, g))
            if op.kind == "int8":
                m, sh = self._requant(op, self.W[-1], self.x[-1])
                self.mult.append(m)
                self.shift.append(sh)
            else:
                self.mult.append(None)
                self.shift.append(None)
            if op.lora_rank:
                A = torch.randn((op.lora_rank, op.cols), generator=g, device=device).mul_(0.02).to(torch.bfloat16)
                B = torch.randn((op.rows, op.lora_rank), generator=g, device=device).mul_(0.02).to(torch.bfloat16)
                ws = torch.empty(op.lora_rank * n_vec, dtype=torch.float32, device=device)
                self.lora.append((A, B, ws))
            else:
                self.lora.append(None)
            if op.epi == "combine":
                rw = torch.rand((n_vec, op.n_active), generator=g, device=device).add_(0.05)
                self.comb.append(rw.div_(rw.sum(dim=1, keepdim=True)))
            else:
                self.comb.append(None)
        torch.cuda.synchronize()
        self.weight_bytes = sum(op.weight_bytes() for op in self.ops)
        self.alg_bytes = [op.alg_bytes(n_vec) for op in self.ops]
        self.x_bytes = int(self.x_all.numel()) * self.x_all.element_size()
        self.ids_bytes = int(ni) * 4
        self.y_bytes = int(self.y_all.numel()) * self.y_all.element_size()

    def _stored_bytes(self, op):
        if op.kind == "moe":
            return op.n_experts * weight_bytes(op.fmt, op.rows, op.cols)
        return weight_bytes(op.fmt, op.rows, op.cols)

    def _weights(self, op, g):
        """Quantized weights of one launch: N(0, 0.02) fp32 quantized on the GPU."""
        torch, hq = self.torch, self.hq
        if op.kind == "int8":
            wf = torch.randn((op.rows, op.cols), generator=g, device=self.device, dtype=torch.float32).mul_(0.02)
            wq = torch.empty((op.rows, op.cols), dtype=torch.int8, device=self.device)
            op_scale = torch.empty(op.rows, dtype=torch.float32, device=self.device)
            hq.hq_quantize_i8_rows(wf, wq, op_scale, op.rows, op.cols)
            self._last_scale = op_scale
            return wq
        quant = {"q8_0": hq.hq_quantize_q8_0, "q4_0": hq.hq_quantize_q4_0, "q4_k": hq.hq_quantize_q4_k}[op.fmt]
        rb = weight_bytes(op.fmt, 1, op.cols)
        n_mat = op.n_experts if op.kind == "moe" else 1
        wq = torch.empty((n_mat * op.rows, rb), dtype=torch.uint8, device=self.device)
        for e in range(n_mat):                      # one matrix (expert) at a time bounds the fp32 scratch
            wf = torch.randn((op.rows, op.cols), generator=g, device=self.device, dtype=torch.float32).mul_(0.02)
            quant(wf, wq[e * op.rows:(e + 1) * op.rows], op.rows, op.cols)
            del wf
        return wq

    def _requant(self, op, wq, xq):
        """Per-row (mult, shift) for M = s_w * s_x / s_out, with s_out the 99th
        percentile of |y| / 127 (about 1 % of outputs saturate).  s_x is the
        symmetric per-tensor scale of x ~ U{-127..127} taken as 1/127."""
        torch, hq = self.torch, self.hq
        s_w = self._last_scale.double()
        s_x = 1.0 / 127.0
        acc = xq.view(self.n_vec, op.cols).double() @ wq.double().t()
        yf = acc * s_w[None, :] * s_x
        s_out = float(torch.quantile(yf.abs().flatten().float(), 0.99)) / 127.0
        M = (s_w * s_x / s_out).cpu().numpy().astype(np.float64)
        mult = np.empty(op.rows, dtype=np.int32)
        shift = np.empty(op.rows, dtype=np.int32)
        hq.hq_requant_params(M, op.rows, mult, shift)
        return torch.from_numpy(mult).to(self.device), torch.from_numpy(shift).to(self.device)

    def launch_all(self, stream, events=None):
        hq, n_vec = self.hq, self.n_vec
        for i, op in enumerate(self.ops):
            if events is not None:
                events.record_before(i, stream)
            if op.kind == "dense" and op.lora_rank:
                A, B, ws = self.lora[i]
                fn = hq.hq_matvec_q8_0_lora if op.fmt == "q8_0" else hq.hq_matvec_q4_0_lora
                fn(self.W[i], self.x[i], A, B, LORA_SCALE, op.lora_rank, ws, self.y[i], op.rows, op.cols, n_vec,
                   stream=stream)
            elif op.kind == "dense":
                fn = {"q8_0": hq.hq_matvec_q8_0, "q4_0": hq.hq_matvec_q4_0, "q4_k": hq.hq_matvec_q4_k}[op.fmt]
                fn(self.W[i], self.x[i], self.y[i], op.rows, op.cols, n_vec, stream=stream)
            elif op.kind == "moe":
                # a layer's down launch uses the ids its gate|up launch used: they were written
                # before the launch that precedes it, so its weight copies may start early
                epi = {None: hq.HQ_MOE_EPI_NONE, "swiglu": hq.HQ_MOE_EPI_SWIGLU,
                       "combine": hq.HQ_MOE_EPI_COMBINE}[op.epi]
                flags = hq.HQ_MOE_IDS_READY if op.label == "down" else 0
                hq.hq_moe_matvec_q8_0_ex(self.W[i], self.ids[i], self.x[i], op.x_per_slot, self.comb[i],
                                         self.y[i], op.n_experts, op.n_active, op.rows, op.cols, n_vec, epi,
                                         flags, stream=stream)
            else:
                hq.hq_matvec_i8_requant(self.W[i], self.x[i], self.mult[i], self.shift[i], self.y[i],
                                        op.rows, op.cols, n_vec, stream=stream)
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
        n0 = self.hq.hq_launch_count()
        with torch.cuda.graph(graph, stream=s):
            self.launch_all(torch.cuda.current_stream().cuda_stream, events)
        torch.cuda.synchronize()
        self.launches_per_step = self.hq.hq_launch_count() - n0     # kernels the library put in one step
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
    """The C oracle (one thread) on a bounded sample of the workload, quantized
    by the oracle itself.  One pass = one call per distinct launch shape:
    dense -- the first rows (about 4M weights) of the matrix; MoE -- the first
    layer's routing over a bank of only its distinct experts, each cut to its
    first rows (about 4M weights in all); int8 -- each of the two matrices
    whole (3.1M weights each), with the oracle's own requant recipe."""

    def __init__(self, name, n_vec, seed=synthetic.SEED_BASE + 2):
        import oracle
        self.oracle = oracle
        self.model, self.fmt, ops = workload_ops(name, n_vec)
        self.n_vec = n_vec
        self.kind = ops[0].kind
        distinct, keys = [], set()
        for op in ops:
            k = (op.rows, op.cols, op.x_per_slot, op.epi)
            if k not in keys:
                keys.add(k)
                distinct.append(op)
        g = synthetic.rng(seed)
        self.calls = []
        self.dense = []                            # (blocks, x, rows, cols) of the plain dense calls
        self.pass_bytes = 0
        for op in distinct:
            if op.kind == "dense":
                r = min(op.rows, max(8, (1 << 22) // op.cols))
                W = synthetic.weights(g, r, op.cols)
                blocks = oracle.quantize(self.fmt, W)
                x = synthetic.activations(g, n_vec, op.cols)
                self.calls.append(lambda b=blocks, x=x, r=r, c=op.cols: oracle.matvec(self.fmt, b, x, r, c))
                if not op.lora_rank:
                    self.dense.append((blocks, x, r, op.cols))
                self.pass_bytes += weight_bytes(self.fmt, r, op.cols)
                if op.lora_rank:
                    # the adapter term of the same sampled rows (bf16 bit patterns of N(0, 0.02))
                    A = (g.standard_normal((op.lora_rank, op.cols)).astype(np.float32) * np.float32(0.02)).view(np.uint32) >> 16
                    B = (g.standard_normal((r, op.lora_rank)).astype(np.float32) * np.float32(0.02)).view(np.uint32) >> 16
                    A, B = A.astype(np.uint16), B.astype(np.uint16)
                    self.calls.append(lambda A=A, B=B, x=x: oracle.lora_delta(A, B, x, LORA_SCALE))
                    self.pass_bytes += 2 * op.lora_rank * (r + op.cols)
            elif op.kind == "moe":
                uniq, remap = np.unique(op.ids, return_inverse=True)
                U = len(uniq)
                r = min(op.rows, max(8, (1 << 22) // (op.cols * U)))
                bank = oracle.quantize_q8_0(synthetic.weights(g, U * r, op.cols))
                ids = remap.reshape(op.ids.shape).astype(np.int32)
                x = synthetic.activations(g, n_vec * (op.n_active if op.x_per_slot else 1), op.cols)
                moe = (lambda b=bank, i=ids, x=x, o=op, U=U, r=r:
                       oracle.moe_matvec_q8_0(b, i, x, o.x_per_slot, U, o.n_active, r, o.cols, n_vec))
                if op.epi == "swiglu":
                    self.calls.append(lambda f=moe: oracle.swiglu_pairs(f()[0]))
                elif op.epi == "combine":
                    rw = synthetic.router_weights(g, n_vec, op.n_active)
                    self.calls.append(lambda f=moe, w=rw: oracle.moe_combine(*f(), w))
                else:
                    self.calls.append(moe)
                self.pass_bytes += U * weight_bytes("q8_0", r, op.cols)
            else:
                W = synthetic.weights(g, op.rows, op.cols)
                xf = synthetic.activations(g, n_vec, op.cols)
                Wq, xq, mult, shift = oracle.int8_workload(W, xf)
                self.calls.append(lambda W=Wq, x=xq, m=mult, s=shift: oracle.matvec_i8_requant(W, x, m, s))
                self.pass_bytes += op.rows * op.cols + 8 * op.rows
        self.n_shapes = len(distinct)

    def run_pass(self):
        for c in self.calls:
            c()
        return self.pass_bytes

    def describe(self, passes):
        what = {"dense": "the first rows (~4M weights) of each of the {n} distinct {m} matrix shapes",
                "moe": "the first layer's routing for each of the {n} MoE launch shapes, over a bank of only "
                       "its distinct experts cut to ~4M weights",
                "int8": "each of the {n} int8 matrices whole, oracle requant recipe"}[self.kind]
        return (f"{passes} passes; each = " + what.format(n=self.n_shapes, m=self.model) +
                f", {self.pass_bytes / 1e6:.1f} MB of {self.fmt} weights, n_vec={self.n_vec}, "
                f"single-threaded C oracle (f64 accumulation for the float formats)")

    def timed(self, budget_s):
        done, n, t0 = 0, 0, time.perf_counter()
        while True:
            done += self.run_pass()
            n += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                return done / el / 1e9, self.describe(n), el

    def timed_all_cores(self, budget_s, workers):
        """The same dense sample with each call's rows split over `workers`
        host threads (the C oracle runs with the interpreter lock released, so
        the threads run on separate cores).  None for non-dense workloads."""
        if self.kind != "dense" or not self.dense:
            return None
        import concurrent.futures as cf
        oracle = self.oracle
        jobs = []
        for (blocks, x, r, c) in self.dense:
            bounds = np.linspace(0, r, workers + 1).astype(int)
            jobs += [(blocks, x, r, c, int(lo), int(hi)) for lo, hi in zip(bounds[:-1], bounds[1:]) if hi > lo]
        per_pass = sum(weight_bytes(self.fmt, r, c) for (_, _, r, c) in self.dense)
        done, n, t0 = 0, 0, time.perf_counter()
        with cf.ThreadPoolExecutor(max_workers=workers) as ex:
            while True:
                list(ex.map(lambda j: oracle.matvec_rows(self.fmt, j[0], j[1], j[2], j[3], j[4], j[5]), jobs))
                done += per_pass
                n += 1
                el = time.perf_counter() - t0
                if el >= budget_s:
                    desc = (f"{n} passes; each = the first rows (~4M weights) of each of the {len(self.dense)} "
                            f"distinct {self.model} matrix shapes, {per_pass / 1e6:.1f} MB of {self.fmt} weights, "
                            f"n_vec={self.n_vec}, every call's rows split over {workers} threads of the C oracle "
                            f"(f64 accumulation)")
                    return done / el / 1e9, desc, el


# ----------------------------------------------------------------- sweep

# the benchmark spec's metric's other points, measured in the default run: the same
# 8B decode token at the speculative-verify widths, and in the 4-bit formats
SWEEP = [("8b-q8_0", 2), ("8b-q8_0", 4), ("8b-q8_0", 8), ("8b-q4_0", 1), ("8b-q4_k", 1)]


def roof_of(ops, n_vec, dev_ms, alg_total, peak, sm_mhz, n_sms):
    """Roofline of a step: HBM (bytes against the measured copy bandwidth)
    unless its flops per byte exceed the FP32 ridge, then the FP32 pipe."""
    achieved = alg_total / (dev_ms / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4)}
    flops = fp32_flops(ops, n_vec)
    if flops is not None and sm_mhz:
        fp32_peak = n_sms * 128 * 2 * sm_mhz * 1e6 / 1e12
        if flops / alg_total > fp32_peak * 1e3 / peak:
            tflops = flops / (dev_ms / 1e3) / 1e12
            roof = {"bound": "alu", "achieved": round(tflops, 2), "peak": round(fp32_peak, 1), "unit": "TFLOP/s",
                    "frac": round(tflops / fp32_peak, 4),
                    "peak_basis": f"{n_sms} SMs x 128 FP32 FMA/clk x 2 x {sm_mhz} MHz"}
    return roof


def sweep_entry(workload, n_vec, steps, warmup, device, peak, seed):
    """One point of the sweep: the step's graph replayed `steps` times after
    `warmup`, CUDA events on the replay stream, clocks sampled meanwhile."""
    import torch
    step = Step(workload, n_vec, device, seed)
    graph = step.capture()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(device.index or 0) as clocks:
        e0.record()
        for _ in range(steps):
            graph.replay()
        e1.record()
        e1.synchronize()
    dev_ms = e0.elapsed_time(e1) / steps
    clk = clocks.summary()
    n_sms = torch.cuda.get_device_properties(device).multi_processor_count
    alg = float(sum(step.alg_bytes))
    out = {"workload": workload, "format": step.fmt, "n_vec": n_vec,
           "value": round(step.weight_bytes / (dev_ms / 1e3) / 1e9, 2), "unit": "GB/s",
           "ms_per_step": round(dev_ms, 5), "tok_per_s": round(1e3 / dev_ms * n_vec, 2),
           "roofline": roof_of(step.ops, n_vec, dev_ms, alg, peak, clk.get("sm_mhz"), n_sms),
           "clocks": clk}
    del graph, step
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------- main

def describe_workload(args, model, fmt, ops, kind):
    if args.shape:
        return f"{len(ops)} distinct {args.shape} {fmt} matrices per step, n_vec={args.n_vec}"
    if kind == "dense":
        fused = WORKLOADS[args.workload][3]
        note = " with q|k|v and gate|up row-fused (same input)" if fused else ", every projection its own call"
        lora = (f"; a rank-{LORA_RANK[args.workload]} bf16 QLoRA adapter (scale {LORA_SCALE:g}) on every "
                f"projection, its bytes counted as weights, two kernels per adapted matvec"
                if args.workload in LORA_RANK else "")
        return (f"{model} decode token, {fmt}, n_vec={args.n_vec}: {len(ops)} matvecs "
                f"(all projections + lm_head){note}{lora}")
    if kind == "moe":
        ffn = ("; gate|up rows interleaved with the SwiGLU epilogue, down with the router-weighted sum "
               "over the slots in the same launch" if args.workload in MOE_FFN else "")
        return (f"MoE decode, {MOE_LAYERS} layers x (gate|up 1536x2048 + down 2048x768) per expert, "
                f"128 experts, 8 active per token drawn uniformly per layer, {fmt}, n_vec={args.n_vec}: "
                f"{len(ops)} expert-indexed launches{ffn}")
    return (f"int8 GEMV + per-row requant, {INT8_COPIES} distinct copies of each of 1024x3072 and 3072x1024, "
            f"n_vec={args.n_vec}: {len(ops)} launches")


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
    ap.add_argument("--format", choices=["q8_0", "q4_0", "q4_k"], default="q8_0", help="format for --shape")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the sweep over n_vec and formats that the default 8B Q8_0 run adds")
    ap.add_argument("--traffic-file", default=os.path.join(ROOT, "profiles", "dram_traffic.txt"),
                    help="DRAM bytes per step of the matvec kernel, from an ncu capture (text)")
    args = ap.parse_args()

    world, rank, local_rank = dist_env()
    model, fmt, ops = workload_ops(args.workload, args.n_vec, args.shape, args.format)
    kind = WORKLOADS[args.workload][0] if not args.shape else "dense"
    config = {"workload": describe_workload(args, model, fmt, ops, kind),
              "shape_set": model, "format": fmt, "n_vec": args.n_vec, "launches_per_step": len(ops),
              "l2": (f"inputs larger than L2: every launch reads its own weights, "
                     f"{sum(op.weight_bytes() for op in ops) / 1e9:.2f} GB per step"),
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
                                 "sample": samp.describe(args.steps) + " (one pass per step)",
                                 "cpu": cpu_model()},
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
    launches_per_step = step.launches_per_step
    events = LaunchEvents(len(ops), _cudart())
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
        per_launch = np.zeros(len(ops))
        for _ in range(args.steps):
            graph_ev.replay()
            per_launch += np.array(events.durations_ms())
        per_launch /= args.steps
        # ---- end to end: pinned host x in, y out, every step
        x_host = step.x_all.cpu().pin_memory()
        ids_host = step.ids_all.cpu().pin_memory()
        y_host = torch.empty(step.y_all.shape, dtype=step.y_all.dtype).pin_memory()

        def e2e_step():
            step.x_all.copy_(x_host, non_blocking=True)
            if step.ids_bytes:
                step.ids_all.copy_(ids_host, non_blocking=True)
            graph.replay()
            y_host.copy_(step.y_all, non_blocking=True)
        for _ in range(2):
            e2e_step()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            e2e_step()
        e1.record()
        e1.synchronize()
        e2e_ms = e0.elapsed_time(e1) / args.steps
    clk = clocks.summary()
    # a wait that timed out inside a kernel leaves its mark here: such a run is not a measurement
    import quantized_weight_matvec_hq_gb300 as hq
    fault = hq.hq_device_fault()
    if fault:
        raise SystemExit(f"device fault word {fault:#x} during the timed run")

    if world > 1:
        dev_ms, e2e_ms = max_over_ranks([dev_ms, e2e_ms], device)

    if rank != 0:
        torch.distributed.destroy_process_group()
        return

    peak, peak_kind = load_peaks()
    probe = read_probe_gbs(device)
    value = aggregate_value(world, step.weight_bytes, dev_ms)
    e2e = aggregate_value(world, step.weight_bytes, e2e_ms)
    # Roofline of the matvec kernel: the step consists of its launches only, so
    # the mean launch duration is the step's device time over the launch count.
    # The event pairs of the per-shape breakdown add a few microseconds per
    # launch and break the programmatic-launch overlap: a breakdown only.
    alg = np.array(step.alg_bytes, dtype=np.float64)
    achieved = float(alg.sum() / (dev_ms / 1e3) / 1e9)
    traffic = read_traffic(args.traffic_file, args.workload, args.n_vec, args.shape)
    kernel_ms = float(per_launch.sum())
    by_shape = {}
    for op, ms, b in zip(ops, per_launch, alg):
        k = f"{op.label} {op.rows}x{op.cols}"
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
        "dtype": ("int32 accumulate, int8 requant" if fmt == "i8" else "fp32 accumulate over " + fmt), "data": "synthetic", "config": config,
        "tok_per_s": round(1e3 / dev_ms * world * args.n_vec, 2),     # n_vec tokens (verify width) per step
        "frac_of_hbm": round(value / world / peak, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": (round(traffic / len(ops)) if traffic is not None else None),
                     "traffic_unit": "DRAM bytes read+written per launch (mean over the step), from ncu",
                     "algorithmic_bytes_per_launch": round(float(alg.sum()) / len(ops)),
                     "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs), burst",
                     "kernel": "matvec_tma_kernel (every launch of the step)",
                     "launches_per_step": len(ops),
                     "mean_launch_us": round(dev_ms * 1e3 / len(ops), 3)},
        "hbm_references": {"measured_copy_gbs": peak, "read_probe_gbs": round(probe, 1),
                           "spec_gbs": 8000.0, "frac_of_read_probe": round(achieved / probe, 4),
                           "frac_of_spec": round(achieved / 8000.0, 4),
                           "read_probe": "torch sum over a 2 GiB fp32 buffer, CUDA events, after the timed region"},
        "per_shape_event_pairs": shapes_out,
        "per_shape_event_pairs_ms_per_step": round(kernel_ms, 4),
        "e2e": {"value": round(e2e, 2), "unit": "GB/s", "ms_per_step": round(e2e_ms, 5),
                "h2d_bytes_per_step": int(step.x_bytes + step.ids_bytes), "d2h_bytes_per_step": int(step.y_bytes)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    # FP32 roof: where the step's flops per byte exceed the ridge of the FP32
    # pipe (SMs x 128 FMA lanes x 2 flops x the sampled SM clock) over the HBM
    # copy bandwidth, the FP32 pipe, not HBM, is the lower roof
    flops = fp32_flops(ops, args.n_vec)
    if flops is not None and clk.get("sm_mhz"):
        n_sms = torch.cuda.get_device_properties(device).multi_processor_count
        fp32_peak = n_sms * 128 * 2 * clk["sm_mhz"] * 1e6 / 1e12
        tflops = flops / (dev_ms / 1e3) / 1e12
        line["fp32_roof"] = {"achieved_tflops": round(tflops, 2), "peak_tflops": round(fp32_peak, 1),
                             "frac": round(tflops / fp32_peak, 4),
                             "flops_per_byte": round(flops / float(alg.sum()), 2),
                             "ridge_flops_per_byte": round(fp32_peak * 1e3 / peak, 2),
                             "peak_basis": f"{n_sms} SMs x 128 FP32 FMA/clk x 2 x {clk['sm_mhz']} MHz"}
        if flops / float(alg.sum()) > fp32_peak * 1e3 / peak:
            line["roofline"].update({"bound": "alu", "achieved": round(tflops, 2), "peak": round(fp32_peak, 1),
                                     "unit": "TFLOP/s", "frac": round(tflops / fp32_peak, 4),
                                     "peak_source": line["fp32_roof"]["peak_basis"] +
                                     " (derived from unit counts and the sampled clock)"})
    if fmt in ("q4_0", "q4_k") and args.n_vec <= 2:
        line["roofline"]["limiter"] = ("nibble decode issue rate (one and per weight on the ALU pipe, one ffma2 "
                                       "per two weights on the FMA pipe), not HBM")
    # the rest of the benchmark spec's metric (n_vec 2, 4, 8; Q4_0 and Q4_K at one
    # vector), one GPU, after the headline's buffers are released
    if (world == 1 and not args.no_sweep and not args.shape and args.workload == "8b-q8_0"
            and args.n_vec == 1):
        del graph, graph_ev, step
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        line["sweep"] = [sweep_entry(w, nv, args.steps, args.warmup, device, peak, synthetic.SEED_BASE + 2)
                         for (w, nv) in SWEEP]
    if not args.no_cpu_baseline and not args.shape:
        samp = OracleSample(args.workload, args.n_vec)
        gbs, desc, el = samp.timed(args.cpu_budget)
        line["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "sample": desc, "seconds": round(el, 2), "cpu": cpu_model()}
        workers = os.cpu_count() or 1
        par = samp.timed_all_cores(args.cpu_budget / 2, workers)
        if par is not None:
            line["cpu_baseline_all_cores"] = {"value": round(par[0], 4), "unit": "GB/s", "cores": workers,
                                              "kind": "oracle", "sample": par[1], "seconds": round(par[2], 2),
                                              "cpu": cpu_model()}
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
