"""Measures the three row-reduction strategies of the fused residual +
LayerNorm + affine kernel across hidden widths and prints where each wins:
the data behind the explicit width boundaries of tf_residual_layernorm
("Costs and benefits of kernel fusion", worked example: test a hidden width
large enough to require a different row-reduction strategy; the dispatch
boundary should be explicit rather than inherited from one benchmark shape).

    python -m gemm_conv_epilogues_gb300.ln_sweep [--json out.json] [--widths 24576,32768]
    python -m gemm_conv_epilogues_gb300.ln_sweep --widths 32768 --variant cluster --plain 3

--plain N skips the timing and just launches the chosen strategy N times on
the width's inputs, one call after another (for profiler captures).

For each width the row count is chosen so act + res + y move about 400 MB
(more than three times the L2); each strategy is timed by CUDA-graph replay.
"""
from __future__ import annotations

import argparse
import json
import statistics

import numpy as np
import torch

from . import binding as b
from . import synth

NAMES = {b.TF_LN_WARP: "warp", b.TF_LN_CTA: "cta", b.TF_LN_CLUSTER: "cluster"}
WIDTHS = [128, 256, 512, 768, 1024, 1536, 2048, 4096, 8192, 16384, 24576, 32768, 65536, 131072]


def _time_us(fn, reps: int = 10) -> float:
    fn()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=torch.cuda.Stream()):
        for _ in range(reps):
            fn()
    graph.replay()
    torch.cuda.synchronize()
    out = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1) * 1e3 / reps)
    return statistics.median(out)


def run(widths=WIDTHS):
    rows_out = []
    for h in widths:
        rows = max(1, (400 * 2**20) // (6 * h))
        d = synth.layernorm_inputs(rows, h, seed=0)
        up = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dtype=dt)).cuda()
        act, res = up(d["act"], np.float16), up(d["res"], np.float16)
        g, be = up(d["gamma"], np.float32), up(d["beta"], np.float32)
        y = torch.empty_like(act)
        t = {}
        for v in NAMES:
            if b.tf_residual_layernorm_variant(act, res, g, be, y, rows, h, 1e-5, v, check=False) != b.TF_OK:
                continue
            us = _time_us(lambda v=v: b.tf_residual_layernorm_variant(act, res, g, be, y, rows, h, 1e-5, v))
            t[NAMES[v]] = {"us": us, "GBs": (6 * rows * h + 8 * h) / us / 1e3}
        best = max(t, key=lambda k: t[k]["GBs"])
        rows_out.append({"hidden": h, "rows": rows, "results": t, "best": best,
                         "dispatch": NAMES.get(b.tf_residual_layernorm_select(h), "-")})
        del act, res, y
        torch.cuda.empty_cache()
    rc, word = b.tf_read_device_error()
    if rc != b.TF_OK:
        raise SystemExit(f"device error word {word:#x}")
    return rows_out


def markdown(rows) -> str:
    out = ["| hidden | rows | warp GB/s | cta GB/s | cluster GB/s | fastest | dispatch |", "|---:|---:|---:|---:|---:|---|---|"]
    for r in rows:
        f = lambda k: f"{r['results'][k]['GBs']:.0f}" if k in r["results"] else "-"
        out.append(f"| {r['hidden']} | {r['rows']} | {f('warp')} | {f('cta')} | {f('cluster')} | {r['best']} | "
                   f"{r['dispatch']} |")
    return "\n".join(out)


def plain(h: int, variant: int, calls: int):
    rows = max(1, (400 * 2**20) // (6 * h))
    d = synth.layernorm_inputs(rows, h, seed=0)
    up = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dtype=dt)).cuda()
    act, res = up(d["act"], np.float16), up(d["res"], np.float16)
    g, be = up(d["gamma"], np.float32), up(d["beta"], np.float32)
    y = torch.empty_like(act)
    for _ in range(calls):
        b.tf_residual_layernorm_variant(act, res, g, be, y, rows, h, 1e-5, variant)
    torch.cuda.synchronize()
    rc, word = b.tf_read_device_error()
    if rc != b.TF_OK:
        raise SystemExit(f"device error word {word:#x}")
    print(json.dumps({"hidden": h, "rows": rows, "variant": variant, "calls": calls}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--json", default=None)
    ap.add_argument("--widths", default=None, help="comma-separated hidden widths (default: the full list)")
    ap.add_argument("--variant", default="auto", choices=["auto", "warp", "cta", "cluster"])
    ap.add_argument("--plain", type=int, default=0, help="only launch the variant this many times (profiling)")
    args = ap.parse_args()
    widths = [int(w) for w in args.widths.split(",")] if args.widths else WIDTHS
    if args.plain:
        v = {"auto": b.TF_LN_AUTO, "warp": b.TF_LN_WARP, "cta": b.TF_LN_CTA, "cluster": b.TF_LN_CLUSTER}[args.variant]
        for h in widths:
            plain(h, v, args.plain)
        return
    rows = run(widths)
    if args.json:
        with open(args.json, "w") as f:
            json.dump(rows, f, indent=1)
    print(markdown(rows))


if __name__ == "__main__":
    main()
