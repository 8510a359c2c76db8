"""Benchmark of the epilogue-fusion hot path on GB300.

Headline (the JSON line's `value`): fused conv2d + BN + SiLU on the largest
workload, NHWC bf16 16x64x64x512 -> 512, 7x7, pad 3 (1.684 TFLOP per step),
through the C ABI with every input resident in HBM, in TFLOP/s.  The same run
measures the other workloads of the path -- fused bias + GELU on fp16
[8192, 8192], fused residual + LayerNorm + affine on fp16 [16384, 4096], the
1x1 conv 32x56x56x256 -> 256 and the tiny 3x3 conv -- each next to the
unfused chain of our own separate kernels, and reports them under
`workloads`.

L2: each workload rotates over enough copies of its input/output buffers that
more than twice the 126 MB L2 is touched between two uses of the same buffer,
so every timed step reads its inputs from HBM.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch under torch.distributed.run (one process per GPU); each rank
runs its own replica of the workload (weak scaling, no collective on the data
path) and rank 0 prints the aggregate.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = "conv7x7_16x64x64x512_to512"
METRIC = "conv+BN+SiLU TFLOP/s (% bf16 peak); fused-chain GB/s (% HBM peak)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 126 * 2**20


# ---------------------------------------------------------------- peaks, clocks, traffic

def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            p = json.load(open(path))
            hbm = p.get("hbm_gbs")
            bf16 = p.get("bf16_tflops")
            if hbm and bf16:
                return {"hbm_gbs": float(hbm), "bf16_tflops": float(bf16),
                        "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained") or bf16),
                        "source": "of measured"}
        except Exception:
            pass
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0, "source": "of fallback"}


class ClockSampler:
    """nvidia-smi clock/throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        self.rows = []
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        for row in csv.reader(io.StringIO(out)):
            if len(row) >= 9:
                self.rows.append([c.strip() for c in row])

    def summary(self) -> dict:
        rows = getattr(self, "rows", [])
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def files_fingerprint(files) -> str:
    """Hash of the named kernel sources: a change to any of them invalidates
    the DRAM-traffic figure captured before it."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "gemm_conv_epilogues_gb300", "csrc")
    for f in sorted(files):
        h.update(f.encode())
        h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


def kernel_traffic(workload: str):
    """DRAM bytes (read + write) per launch of the workload's fused kernel from
    the committed ncu summary, if none of the kernel's source files has
    changed since the capture (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        e = json.load(open(path)).get(workload)
        if not e or files_fingerprint(e["files"]) != e["files_sha256_16"]:
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------- distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    """Largest value over the ranks (the slowest rank's time)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_throughput(units_per_rank: float, ms_slowest: float, world: int, scale: float = 1e12) -> float:
    """Weak scaling: every rank processes `units_per_rank`; the job's rate is
    all ranks' units over the slowest rank's time (per second, / scale)."""
    return units_per_rank * world / (ms_slowest * 1e-3) / scale


# ---------------------------------------------------------------- workloads

class Runner:
    """Device buffers of one workload (several rotating sets) and the launch
    functions of its fused call and unfused chain."""

    def __init__(self, name: str, seed: int):
        import torch
        from gemm_conv_epilogues_gb300 import binding as b, synth
        self.b, self.torch = b, torch
        self.w = synth.WORKLOADS[name]
        self.name = name
        self.inputs = synth.workload_inputs(self.w, seed)
        d = self.inputs
        dev = "cuda"
        up16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16).copy()).to(dev)
        up = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dtype=dt).copy()).to(dev)
        w = self.w
        if w.kind == "conv":
            c = w.conv
            self.shape = b.conv_shape(c.N, c.H, c.W, c.C_in, c.C_out, c.KH, c.KW, c.stride, c.pad)
            self.M = c.M
            self.flops = c.flops
            x_bytes = c.N * c.H * c.W * c.C_in * 2
            y_bytes = c.M * c.C_out * 2
            w_bytes = c.C_out * c.K * 2
            self.alg_bytes = x_bytes + y_bytes + w_bytes + 8 * c.C_out
            self.unfused_extra = 4 * y_bytes
            self.h2d, self.d2h = x_bytes, y_bytes
            self.wt = torch.empty((c.C_out, c.KH, c.KW, c.C_in), dtype=torch.int16, device=dev)
            b.tf_pack_filter_nhwc(up16(d["w_oihw"]), self.wt, c.C_out, c.C_in, c.KH, c.KW)   # load time
            self.scale, self.bias = up(d["scale"], np.float32), up(d["bias"], np.float32)
            per_set = x_bytes + y_bytes
            nsets = max(1, min(8, int(np.ceil(2 * L2_BYTES / per_set)) + 1))
            x0 = up16(d["x"])
            self.sets = []
            for _ in range(nsets):
                self.sets.append({"x": x0.clone(), "y": torch.empty((c.M, c.C_out), dtype=torch.int16, device=dev)})
            self.t1 = torch.empty((c.M, c.C_out), dtype=torch.int16, device=dev)
            self.t2 = torch.empty_like(self.t1)
            self.host_x = torch.from_numpy(d["x"].view(np.int16).copy()).pin_memory()
            self.host_y = torch.empty((c.M, c.C_out), dtype=torch.int16).pin_memory()
        elif w.kind in ("bias_gelu", "bias_gelu_rowsum"):
            rows, cols = w.rows, w.cols
            self.flops = 0
            n = rows * cols
            self.alg_bytes = 2 * n + 2 * n + 2 * cols + (4 * rows if w.kind == "bias_gelu_rowsum" else 0)
            # split paths: the x + bias intermediate (write + read), or the re-read of y by the reduction
            self.unfused_extra = 4 * n if w.kind == "bias_gelu" else 2 * n
            self.rowsum = torch.empty((rows,), dtype=torch.float32, device=dev)
            self.h2d, self.d2h = 2 * n, 2 * n
            per_set = 4 * n
            nsets = max(1, int(np.ceil(2 * L2_BYTES / per_set)) + 1)
            x0 = up(d["x"], np.float16)
            self.bias = up(d["bias"], np.float16)
            self.sets = [{"x": x0.clone(), "y": torch.empty_like(x0)} for _ in range(nsets)]
            self.t = torch.empty_like(x0)
            self.host_x = torch.from_numpy(d["x"].copy()).pin_memory()
            self.host_y = torch.empty((rows, cols), dtype=torch.float16).pin_memory()
        else:
            rows, hidden = w.rows, w.cols
            self.flops = 0
            n = rows * hidden
            self.alg_bytes = 2 * n * 3 + 8 * hidden
            self.unfused_extra = 8 * n
            self.h2d, self.d2h = 4 * n, 2 * n
            per_set = 6 * n
            nsets = max(1, int(np.ceil(2 * L2_BYTES / per_set)) + 1)
            a0, r0 = up(d["act"], np.float16), up(d["res"], np.float16)
            self.gamma, self.beta = up(d["gamma"], np.float32), up(d["beta"], np.float32)
            self.sets = [{"a": a0.clone(), "r": r0.clone(), "y": torch.empty_like(a0)} for _ in range(nsets)]
            self.s = torch.empty_like(a0)
            self.n = torch.empty_like(a0)
            self.host_a = torch.from_numpy(d["act"].copy()).pin_memory()
            self.host_r = torch.from_numpy(d["res"].copy()).pin_memory()
            self.host_y = torch.empty((rows, hidden), dtype=torch.float16).pin_memory()
        self.nsets = len(self.sets)

    # one fused call on buffer set i (time_loop counts the kernels it launches
    # with the library's own launch counter)
    def fused(self, i: int) -> None:
        b, s, w = self.b, self.sets[i % self.nsets], self.w
        if w.kind == "conv":
            b.tf_conv2d_bn_silu(s["x"], self.wt, self.scale, self.bias, s["y"], self.shape)
        elif w.kind == "bias_gelu":
            b.tf_bias_gelu(s["x"], self.bias, s["y"], w.rows, w.cols)
        elif w.kind == "bias_gelu_rowsum":
            b.tf_bias_gelu_rowsum(s["x"], self.bias, s["y"], self.rowsum, w.rows, w.cols)
        else:
            b.tf_residual_layernorm(s["a"], s["r"], self.gamma, self.beta, s["y"], w.rows, w.cols, w.eps)

    def unfused(self, i: int) -> None:
        b, s, w = self.b, self.sets[i % self.nsets], self.w
        if w.kind == "conv":
            c = w.conv
            b.tf_unfused_conv2d(s["x"], self.wt, self.t1, self.shape)
            b.tf_unfused_bn(self.t1, self.scale, self.bias, self.t2, c.M, c.C_out)
            b.tf_unfused_silu(self.t2, s["y"], c.M * c.C_out)
            return
        if w.kind == "bias_gelu":
            b.tf_unfused_bias_add(s["x"], self.bias, self.t, w.rows, w.cols)
            b.tf_unfused_gelu(self.t, s["y"], w.rows * w.cols)
            return
        if w.kind == "bias_gelu_rowsum":
            b.tf_bias_gelu(s["x"], self.bias, s["y"], w.rows, w.cols)
            b.tf_unfused_rowsum(s["y"], self.rowsum, w.rows, w.cols)
            return
        b.tf_unfused_residual_add(s["a"], s["r"], self.s, w.rows * w.cols)
        b.tf_unfused_layernorm(self.s, self.n, w.rows, w.cols, w.eps)
        b.tf_unfused_affine(self.n, self.gamma, self.beta, s["y"], w.rows, w.cols)

    # end to end through the C ABI from pinned host buffers: H2D of the step's
    # inputs, the fused call, D2H of the result
    def e2e(self, i: int) -> None:
        s = self.sets[i % self.nsets]
        if self.w.kind == "layernorm":
            s["a"].copy_(self.host_a, non_blocking=True)
            s["r"].copy_(self.host_r, non_blocking=True)
        else:
            s["x"].copy_(self.host_x, non_blocking=True)
        self.fused(i)
        self.host_y.copy_(s["y"].view(self.host_y.shape), non_blocking=True)


def time_e2e_pipelined(r: "Runner", steps: int, warmup: int, world: int) -> float:
    """End-to-end ms per step through the C ABI from pinned host memory: each
    step copies its input host->device, runs the fused call and copies the
    output device->host.  Copies run on their own streams, so step i+1's input
    upload and step i-1's download overlap step i's kernel -- how a caller
    would stream batches; every step still pays for its own copies."""
    import torch
    cur = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    n = r.nsets
    hosts = [r.host_y, torch.empty_like(r.host_y).pin_memory()]
    ev = lambda: torch.cuda.Event()
    total = warmup + steps
    h2d_done, comp_done, d2h_done = [ev() for _ in range(total)], [ev() for _ in range(total)], \
        [ev() for _ in range(total)]
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(total):
        if i == warmup:
            cur.wait_event(d2h_done[i - 1]) if i > 0 else None
            t0.record(cur)
            up.wait_stream(cur)
        s = r.sets[i % n]
        with torch.cuda.stream(up):
            if i >= n:
                up.wait_event(comp_done[i - n])          # the compute that read this input set is done
            s["x"].copy_(r.host_x, non_blocking=True)
            h2d_done[i].record(up)
        cur.wait_event(h2d_done[i])
        if i >= n:
            cur.wait_event(d2h_done[i - n])              # this output set has been downloaded
        r.fused(i)
        comp_done[i].record(cur)
        with torch.cuda.stream(down):
            down.wait_event(comp_done[i])
            hosts[i % 2].copy_(s["y"].view(r.host_y.shape), non_blocking=True)
            d2h_done[i].record(down)
    cur.wait_event(d2h_done[total - 1])
    t1.record(cur)
    torch.cuda.synchronize()
    barrier(world)
    return max_over_ranks(t0.elapsed_time(t1) / steps, world)


class PairRunner:
    """Producer -> consumer convs with the activation between them either in
    the producer's epilogue (fused) or as standalone kernels (BN, then SiLU)
    between a plain producer conv and the consumer."""

    def __init__(self, seed: int):
        import torch
        from gemm_conv_epilogues_gb300 import binding as b, synth
        self.b = b
        p, c = synth.PAIR_PRODUCER, synth.PAIR_CONSUMER
        self.p, self.c = p, c
        d = synth.producer_consumer_inputs(p, c, seed)
        dev = "cuda"
        up16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16).copy()).to(dev)
        up = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)
        self.w1 = torch.empty((p.C_out, p.KH, p.KW, p.C_in), dtype=torch.int16, device=dev)
        self.w2 = torch.empty((c.C_out, c.KH, c.KW, c.C_in), dtype=torch.int16, device=dev)
        b.tf_pack_filter_nhwc(up16(d["w1_oihw"]), self.w1, p.C_out, p.C_in, p.KH, p.KW)
        b.tf_pack_filter_nhwc(up16(d["w2_oihw"]), self.w2, c.C_out, c.C_in, c.KH, c.KW)
        self.s1, self.b1, self.s2, self.b2 = up(d["scale1"]), up(d["bias1"]), up(d["scale2"]), up(d["bias2"])
        self.sh1 = b.conv_shape(p.N, p.H, p.W, p.C_in, p.C_out, p.KH, p.KW, p.stride, p.pad)
        self.sh2 = b.conv_shape(c.N, c.H, c.W, c.C_in, c.C_out, c.KH, c.KW, c.stride, c.pad)
        x_bytes = p.N * p.H * p.W * p.C_in * 2
        u_bytes = p.M * p.C_out * 2
        nsets = max(1, int(np.ceil(2 * L2_BYTES / (x_bytes + 2 * u_bytes))) + 1)
        x0 = up16(d["x"])
        self.sets = [{"x": x0.clone(), "u": torch.empty((p.M, p.C_out), dtype=torch.int16, device=dev),
                      "y": torch.empty((c.M, c.C_out), dtype=torch.int16, device=dev)} for _ in range(nsets)]
        self.t = torch.empty((p.M, p.C_out), dtype=torch.int16, device=dev)
        self.t2 = torch.empty_like(self.t)
        self.nsets = nsets
        self.u_elems = p.M * p.C_out

    def fused(self, i):
        b, s = self.b, self.sets[i % self.nsets]
        b.tf_conv2d_bn_silu(s["x"], self.w1, self.s1, self.b1, s["u"], self.sh1)
        b.tf_conv2d_bn_silu(s["u"], self.w2, self.s2, self.b2, s["y"], self.sh2)

    def standalone(self, i):
        b, s = self.b, self.sets[i % self.nsets]
        b.tf_unfused_conv2d(s["x"], self.w1, self.t, self.sh1)
        self.activation(i)
        b.tf_conv2d_bn_silu(s["u"], self.w2, self.s2, self.b2, s["y"], self.sh2)

    def activation(self, i):
        b, s = self.b, self.sets[i % self.nsets]
        b.tf_unfused_bn(self.t, self.s1, self.b1, self.t2, self.p.M, self.p.C_out)
        b.tf_unfused_silu(self.t2, s["u"], self.u_elems)


def time_loop(fn, steps: int, warmup: int, world: int, clocks=None):
    """Times exactly `steps` calls of fn(i) with CUDA events on the current
    stream, bracketed by a barrier and a device synchronise on both sides;
    returns (max-over-ranks ms per step, kernels launched in the timed region:
    the library's own launch counter, read on both sides of the timed calls)."""
    import torch
    from gemm_conv_epilogues_gb300 import binding as b
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ctx = clocks if clocks is not None else _Null()
    with ctx:
        c0 = b.tf_launch_count()
        ev0.record(stream)
        for i in range(steps):
            fn(warmup + i)
        ev1.record(stream)
        launches = b.tf_launch_count() - c0
        torch.cuda.synchronize()
    barrier(world)
    ms = ev0.elapsed_time(ev1) / steps
    return max_over_ranks(ms, world), launches


def time_alternating(fa, fb, steps: int, warmup: int, world: int, blocks: int = 3):
    """Times fa and fb in alternating blocks of `steps` calls (a, b, a, b, ...),
    each block by time_loop, and returns the median ms per call of each.  On a
    power-capped GPU the clock depends on how long the load has lasted, so the
    two sides of a comparison are measured over the same windows."""
    import statistics
    ta, tb = [], []
    for k in range(blocks):
        ta.append(time_loop(fa, steps, warmup, world)[0])
        tb.append(time_loop(fb, steps, warmup, world)[0])
    return statistics.median(ta), statistics.median(tb)


def graph_time_us(fn, calls: int) -> float:
    """GPU time per call with `calls` calls captured in one CUDA graph and
    replayed, so the host's per-call launch cost is not counted."""
    import torch
    fn(0)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        for i in range(calls):
            fn(i)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / calls


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def copy_reference_gbs(nbytes: int = 1 << 30, reps: int = 20) -> float:
    """Bytes moved per second (read + write) by a plain device-to-device copy
    of `nbytes` through torch: context for the memory-bound kernels' GB/s,
    not a roofline denominator."""
    import torch
    src = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    dst = torch.empty_like(src)
    for _ in range(3):
        dst.copy_(src)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        dst.copy_(src)
    e1.record()
    torch.cuda.synchronize()
    gbs = 2 * nbytes * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9
    del src, dst
    torch.cuda.empty_cache()
    return gbs


def traffic_ratio(workload: str, alg_bytes: int):
    """ncu DRAM bytes per launch over the algorithmic bytes (None without a
    current capture)."""
    t = kernel_traffic(workload)
    return round(t / alg_bytes, 3) if t else None


def roofline(bound, achieved, peak, unit, traffic):
    return {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": traffic}


# ---------------------------------------------------------------- CPU baseline (the oracle)

def cpu_oracle_full(r: "Runner") -> dict:
    """The fp64 oracle, as it stands, on the whole of a (small or memory-bound)
    workload's seeded inputs, on every host core: the baseline the GPU kernel
    sits beside, in the same units."""
    import oracle
    d, w = r.inputs, r.w
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    if w.kind == "conv":
        c = w.conv
        oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], c.stride, c.pad, nthreads=threads)
    elif w.kind == "bias_gelu":
        oracle.bias_gelu(d["x"], d["bias"], nthreads=threads)
    elif w.kind == "bias_gelu_rowsum":
        oracle.bias_gelu_rowsum(d["x"], d["bias"], nthreads=threads)
    else:
        oracle.residual_layernorm(d["act"], d["res"], d["gamma"], d["beta"], eps=1e-5, nthreads=threads)
    dt = time.perf_counter() - t0
    out = {"kind": "oracle", "cores": threads, "sample": "the whole workload", "seconds": round(dt, 3),
           "gbs": round(r.alg_bytes / dt / 1e9, 3)}
    if r.flops:
        out["tflops"] = r.flops / dt / 1e12
    return out


_HEADLINE_INPUTS = {}


def cpu_baseline_conv7x7(target_s: float = 12.0) -> dict:
    """The fp64 oracle, as it stands, on a sample of output pixels of the 7x7
    workload (all 512 channels of each), on every host core.  The seeded
    inputs are generated once per process."""
    import oracle
    from gemm_conv_epilogues_gb300 import synth
    w = synth.WORKLOADS[HEADLINE]
    c = w.conv
    if HEADLINE not in _HEADLINE_INPUTS:
        _HEADLINE_INPUTS[HEADLINE] = synth.workload_inputs(w)
    d = _HEADLINE_INPUTS[HEADLINE]
    threads = oracle.default_threads()
    rng = np.random.default_rng(0)
    flops_per_point = 2 * c.K
    # calibrate on a small sample, then size the timed sample to ~target_s
    pix = rng.integers(0, c.M, 8)
    pts = (pix[:, None] * c.C_out + np.arange(c.C_out)[None, :]).reshape(-1)
    t0 = time.perf_counter()
    oracle.conv2d_bn_silu_points(d["x"], d["w_oihw"], d["scale"], d["bias"], pts, c.stride, c.pad, nthreads=threads)
    rate = pts.size * flops_per_point / (time.perf_counter() - t0)
    npix = int(max(16, min(4096, target_s * rate / (flops_per_point * c.C_out))))
    pix = rng.integers(0, c.M, npix)
    pts = (pix[:, None] * c.C_out + np.arange(c.C_out)[None, :]).reshape(-1)
    t0 = time.perf_counter()
    oracle.conv2d_bn_silu_points(d["x"], d["w_oihw"], d["scale"], d["bias"], pts, c.stride, c.pad, nthreads=threads)
    dt = time.perf_counter() - t0
    tflops = pts.size * flops_per_point / dt / 1e12
    return {"value": tflops, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{npix} random output pixels x all {c.C_out} channels of {HEADLINE} "
                      f"({pts.size * flops_per_point / 1e9:.1f} GFLOP, {dt:.1f} s, fp64 7-loop direct conv)",
            "seconds": dt}


# ---------------------------------------------------------------- main

def run_reference(args, world, rank):
    if rank != 0:
        return
    # every step is a bounded sample sized so that the whole run stays within
    # about two minutes of oracle time, whatever --steps is
    per_step = []
    step_s = min(30.0, max(0.05, 120.0 / max(args.steps, 1)))
    for _ in range(args.warmup):
        cpu_baseline_conv7x7(target_s=min(step_s, 1.0))
    for _ in range(args.steps):
        per_step.append(cpu_baseline_conv7x7(target_s=step_s))
    print(json.dumps(reference_line(per_step, args.gpus, args.steps, args.warmup)), flush=True)


def reference_line(per_step, gpus, steps, warmup) -> dict:
    """The reference arm's JSON line from its timed oracle samples."""
    v = statistics.median(p["value"] for p in per_step)
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": gpus,
            "steps": steps, "warmup": warmup,
            "ms_per_step": statistics.median(p["seconds"] for p in per_step) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": HEADLINE, "note": "bounded sample per step"},
            "cpu_baseline": {"kind": "oracle", "cores": per_step[0]["cores"], "sample": per_step[0]["sample"],
                             "value": v, "unit": "TFLOP/s"},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=600)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only-headline", action="store_true")
    ap.add_argument("--sub-steps", type=int, default=200,
                    help="timed steps of each secondary workload (the tiny conv runs 10x as many)")
    ap.add_argument("--profile-workload", default=None,
                    help="only run W+K fused calls of this workload (for profiler captures)")
    ap.add_argument("--profile-unfused", action="store_true",
                    help="with --profile-workload: run the unfused chain instead of the fused call")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_env()

    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import torch
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from gemm_conv_epilogues_gb300 import build as gbuild
    if rank == 0:
        gbuild.build_library()
    barrier(world)
    from gemm_conv_epilogues_gb300 import binding as b

    if args.profile_workload:
        r = Runner(args.profile_workload, seed=rank)
        fn = r.unfused if args.profile_unfused else r.fused
        for i in range(args.warmup + args.steps):
            fn(i)
        torch.cuda.synchronize()
        rc, word = b.tf_read_device_error()
        if rc != b.TF_OK:
            raise SystemExit(f"device error word {word:#x}")
        print(json.dumps({"profile_workload": args.profile_workload, "calls": args.warmup + args.steps}))
        return

    peaks = load_peaks()
    head = Runner(HEADLINE, seed=rank)
    clocks = ClockSampler(local)
    ms, launches = time_loop(head.fused, args.steps, args.warmup, world, clocks)
    value = whole_job_throughput(head.flops, ms, world)
    per_launch_tflops = head.flops / (ms * 1e-3) / 1e12
    e2e_ms = time_e2e_pipelined(head, max(10, args.steps // 10), args.warmup, world)
    e2e_val = whole_job_throughput(head.flops, e2e_ms, world)
    # the same copies and call with nothing overlapped: copy in, conv, copy out, one after another
    e2e_serial_ms, _ = time_loop(head.e2e, max(5, args.steps // 20), args.warmup, world)
    e2e_serial_val = whole_job_throughput(head.flops, e2e_serial_ms, world)
    rc, word = b.tf_read_device_error()
    if rc != b.TF_OK:
        raise SystemExit(f"device error word {word:#x} after the timed region")

    # Every workload's numbers, compact (the full line stays short enough to be
    # kept whole in a log tail).  Keys: ms = fused ms per call; gbs / tflops =
    # throughput of the algorithmic bytes / flops; frac = fraction of the
    # roofline peak named in `peaks`; dram_ratio = ncu DRAM bytes (read +
    # write, steady state) over the algorithmic bytes; unf_ms = the unfused
    # chain of our own kernels, timed in alternating blocks with the fused
    # call (fused_ms_alt = the fused call in those same windows); cpu_s = the
    # oracle on the whole workload, all host cores.
    workloads = {}
    cmp_steps = max(20, args.steps // 10)
    f_cmp_ms, unf_ms = time_alternating(head.fused, head.unfused, cmp_steps, args.warmup, world)
    head_roof = roofline("tensor", per_launch_tflops, peaks["bf16_tflops"], "TFLOP/s", kernel_traffic(HEADLINE))
    workloads[HEADLINE] = {"ms": round(ms, 5), "tflops": round(per_launch_tflops, 1), "frac": head_roof["frac"],
                           "dram_ratio": traffic_ratio(HEADLINE, head.alg_bytes),
                           "unf_ms": round(unf_ms, 5), "fused_ms_alt": round(f_cmp_ms, 5)}
    del head
    torch.cuda.empty_cache()

    if not args.only_headline:
        for name in ["conv1x1_32x56x56x256_to256", "bias_gelu_f16_8192x8192", "bias_gelu_rowsum_f16_8192x8192",
                     "residual_layernorm_f16_16384x4096", "conv3x3_tiny_1x16x16x8_to16"]:
            r = Runner(name, seed=rank)
            steps = args.sub_steps if r.w.kind != "conv" or r.w.conv.M > 1000 else 10 * args.sub_steps
            f_ms, u_ms = time_alternating(r.fused, r.unfused, steps, args.warmup, world)
            gbs = r.alg_bytes / (f_ms * 1e-3) / 1e9
            entry = {"ms": round(f_ms, 5), "gbs": round(gbs, 1)}
            if name.startswith("conv3x3_tiny"):
                # launch-latency bound (0.59 MFLOP): GPU time per call inside a CUDA graph
                entry["graph_us"] = round(graph_time_us(r.fused, 200), 2)
                entry["unf_graph_us"] = round(graph_time_us(r.unfused, 200), 2)
            else:
                entry["frac"] = round(gbs / peaks["hbm_gbs"], 4)
                entry["dram_ratio"] = traffic_ratio(name, r.alg_bytes)
            if r.flops and not name.startswith("conv3x3_tiny"):
                # a conv below the ridge point: its share of the dense tensor peak
                # next to its share of what the HBM roofline allows at its
                # arithmetic intensity, min(peak, flops/bytes * bandwidth)
                tflops = r.flops / (f_ms * 1e-3) / 1e12
                attainable = min(peaks["bf16_tflops"], r.flops / r.alg_bytes * peaks["hbm_gbs"] / 1e3)
                entry.update({"tflops": round(tflops, 1), "frac_tensor": round(tflops / peaks["bf16_tflops"], 4),
                              "frac_attainable": round(tflops / attainable, 4)})
                if r.w.conv.KH == 1 and r.w.conv.KW == 1:
                    # what a plain device-to-device copy of the same x -> y bytes,
                    # over the same rotating sets, takes: the practical bound at
                    # this transfer size
                    def copy(i, r=r):
                        s = r.sets[i % r.nsets]
                        s["y"].view(-1)[: s["x"].numel()].copy_(s["x"].view(-1))
                    c_ms, _ = time_loop(copy, steps, args.warmup, world)
                    entry["copy_ms"] = round(c_ms, 5)
            entry["unf_ms"] = round(u_ms, 5)
            if rank == 0 and world == 1 and not args.no_cpu_baseline:
                entry["cpu_s"] = cpu_oracle_full(r)["seconds"]
            workloads[name] = entry
            del r
            torch.cuda.empty_cache()

        # the activation between two convs (producer 1x1 256->128, consumer 7x7
        # 128->128 on 16x64x64): in the producer's epilogue, or as standalone
        # BN and SiLU kernels after a plain producer conv
        pr = PairRunner(seed=rank)
        steps = max(10, args.sub_steps // 4)
        f_ms, _ = time_loop(pr.fused, steps, args.warmup, world)
        s_ms, _ = time_loop(pr.standalone, steps, args.warmup, world)
        a_ms, _ = time_loop(pr.activation, steps, args.warmup, world)
        workloads["producer_consumer_1x1_256to128_then_7x7_128to128"] = {
            "ms": round(f_ms, 5), "standalone_ms": round(s_ms, 5), "act_ms": round(a_ms, 5),
            "act_share": round(a_ms / s_ms, 4)}
        del pr
        torch.cuda.empty_cache()
        # a plain 1 GiB device-to-device copy: what streaming reaches on this GPU
        workloads["hbm_copy_reference"] = {"gbs": round(copy_reference_gbs(), 1)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_conv7x7()
        cpu.pop("seconds", None)

    if rank == 0:
        cs = clocks.summary()
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": HEADLINE, "N": 16, "H": 64, "W": 64, "C_in": 512, "C_out": 512, "KH": 7,
                       "KW": 7, "stride": 1, "pad": 3, "flops_per_step_per_gpu": head_flops(),
                       "l2": "rotating input/output buffer sets, >2x L2 touched between reuses",
                       "parallelism": f"replicas x{world}"},
            "roofline": head_roof,
            "peaks": {"hbm_gbs": peaks["hbm_gbs"], "bf16_tflops": peaks["bf16_tflops"],
                      "source": peaks["source"]},
            "e2e": {"value": round(e2e_val, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": int(16 * 64 * 64 * 512 * 2),
                    "d2h_bytes_per_step": int(16 * 64 * 64 * 512 * 2),
                    "mode": "copies on side streams overlap neighbouring steps",
                    "serial_value": round(e2e_serial_val, 2), "serial_ms_per_step": round(e2e_serial_ms, 5)},
            "gpu_launches": launches,
            "clocks": {"sm_mhz": cs["sm_mhz"], "sm_max_mhz": cs["sm_max_mhz"], "reasons": cs["reasons"]},
            "cpu_baseline": cpu,
            "workloads": workloads,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def head_flops() -> int:
    from gemm_conv_epilogues_gb300 import synth
    return synth.WORKLOADS[HEADLINE].conv.flops


if __name__ == "__main__":
    main()
