"""Measures the three conv+BN+SiLU kernels across shapes on the current GPU and
prints which one wins where: the data behind the shape thresholds of
tf_conv2d_bn_silu's kernel choice ("Fusing an Epilogue", "Three kernels for
one operation": hand-picked thresholds are normal, and a bench exists to
check that they still hold).

    python -m gemm_conv_epilogues_gb300.dispatch_sweep [--quick] [--json out.json]

Every variant is timed with CUDA events around replays of a CUDA graph of
back-to-back calls (median of 5 replays), so the numbers are GPU time, not
host launch cost; shapes a variant cannot take are skipped.  "umma+splitk"
is tf_conv2d_bn_silu_ws with a full workspace, for shapes it splits.  The last
column is the kernel the library's dispatch picks today, so a row where it
differs from the fastest one shows a threshold to revisit.
"""
from __future__ import annotations

import argparse
import itertools
import json
import statistics

import numpy as np
import torch

from . import binding as b
from . import synth

NAMES = {b.TF_CONV_DIRECT: "direct", b.TF_CONV_TILED: "tiled", b.TF_CONV_UMMA: "umma",
         b.TF_CONV_UMMA_PAIR: "umma pair", b.TF_CONV_UMMA_PAIR_WIDE: "umma pair, wide tiles",
         b.TF_CONV_UMMA_WIDE: "umma, wide tiles"}


def _time_us(fn, reps: int) -> float:
    """GPU time per call: `reps` calls captured once in a CUDA graph and
    replayed, so the host's per-call launch cost does not hide small kernels."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
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


def shapes(quick: bool):
    couts = [8, 16, 20, 32, 48, 64, 128, 256]
    cins = [8, 24, 64, 256] if not quick else [8, 64]
    spatial = [(1, 16, 16), (4, 32, 32), (16, 64, 64)] if not quick else [(1, 16, 16), (4, 32, 32)]
    kernels = [(1, 0), (3, 1)]
    for co, ci, (n, h, w), (k, p) in itertools.product(couts, cins, spatial, kernels):
        yield synth.ConvShape(n, h, w, ci, co, k, k, (1, 1), (p, p))
    if not quick:   # long reductions (up to the 7x7 workload's 25088)
        for co, (k, p) in itertools.product([128, 256, 512], [(3, 1), (7, 3)]):
            yield synth.ConvShape(16, 64, 64, 512, co, k, k, (1, 1), (p, p))


def run(quick: bool = False):
    rows = []
    dev = "cuda"
    for c in shapes(quick):
        d = synth.conv_inputs(c, seed=0, w_dist="normal_fanin")
        x = torch.from_numpy(d["x"].view(np.int16).copy()).to(dev)
        w = torch.empty((c.C_out, c.KH, c.KW, c.C_in), dtype=torch.int16, device=dev)
        b.tf_pack_filter_nhwc(torch.from_numpy(d["w_oihw"].view(np.int16).copy()).to(dev), w, c.C_out, c.C_in,
                              c.KH, c.KW)
        sc = torch.from_numpy(d["scale"]).to(dev)
        bi = torch.from_numpy(d["bias"]).to(dev)
        y = torch.empty((c.M, c.C_out), dtype=torch.int16, device=dev)
        shape = b.conv_shape(c.N, c.H, c.W, c.C_in, c.C_out, c.KH, c.KW, c.stride, c.pad)
        reps = 20 if c.flops < 1e9 else 5
        t = {}
        for v in (b.TF_CONV_DIRECT, b.TF_CONV_TILED, b.TF_CONV_UMMA, b.TF_CONV_UMMA_PAIR, b.TF_CONV_UMMA_PAIR_WIDE,
                  b.TF_CONV_UMMA_WIDE):
            if b.tf_conv2d_bn_silu_variant(x, w, sc, bi, y, shape, v, check=False) != b.TF_OK:
                continue
            t[NAMES[v]] = _time_us(lambda v=v: b.tf_conv2d_bn_silu_variant(x, w, sc, bi, y, shape, v), reps)
        need = b.tf_conv2d_bn_silu_workspace_size(shape)
        if need > 0:
            ws = torch.empty((need // 4,), dtype=torch.float32, device=dev)
            t["umma+splitk"] = _time_us(lambda: b.tf_conv2d_bn_silu_ws(x, w, sc, bi, y, shape, ws, need), reps)
        rows.append({"N": c.N, "H": c.H, "W": c.W, "C_in": c.C_in, "C_out": c.C_out, "K": c.KH,
                     "M": c.M, "mflop": c.flops / 1e6, "us": t, "best": min(t, key=t.get),
                     "dispatch": NAMES[b.tf_conv2d_bn_silu_select(shape)]})
    rc, word = b.tf_read_device_error()
    if rc != b.TF_OK:
        raise SystemExit(f"device error word {word:#x}")
    return rows


def markdown(rows) -> str:
    out = ["| N,H,W | C_in | C_out | k | MFLOP | direct us | tiled us | umma us | pair us | pair wide us | wide us "
           "| umma+splitk us | fastest | dispatch | dispatch / fastest |",
           "|---|---:|---:|---:|---:|---:|---:|---:|---:|---:|---:|---:|---|---|---:|"]
    for r in rows:
        f = lambda k: f"{r['us'][k]:.1f}" if k in r["us"] else "-"
        # the dispatch never uses a workspace: compare it with the best kernel that needs none
        plain = {k: v for k, v in r["us"].items() if k != "umma+splitk"}
        ratio = plain[r["dispatch"]] / min(plain.values()) if r["dispatch"] in plain else float("nan")
        out.append(f"| {r['N']},{r['H']},{r['W']} | {r['C_in']} | {r['C_out']} | {r['K']} | {r['mflop']:.1f} | "
                   f"{f('direct')} | {f('tiled')} | {f('umma')} | {f('umma pair')} | {f('umma pair, wide tiles')} | "
                   f"{f('umma, wide tiles')} | "
                   f"{f('umma+splitk')} | {r['best']} | {r['dispatch']} | {ratio:.2f} |")
    agree = sum(r["best"] == r["dispatch"] for r in rows)
    out.append(f"\ndispatch picks the fastest kernel in {agree} of {len(rows)} shapes")
    return "\n".join(out)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--quick", action="store_true")
    ap.add_argument("--json", default=None)
    args = ap.parse_args()
    torch.cuda.init()
    rows = run(args.quick)
    if args.json:
        with open(args.json, "w") as f:
            json.dump(rows, f, indent=1)
    print(markdown(rows))


if __name__ == "__main__":
    main()
