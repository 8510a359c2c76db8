"""Seeded synthetic inputs, shared by the tests, the smoke check and the bench.

This module holds none of the method's arithmetic: it only draws random
numbers, rounds them to the storage formats (bf16 / fp16, round to nearest
even) and names the workload shapes.  Both the CUDA path and the oracle
receive the very same bits from here.

Generator: numpy's PCG64 bit generator, one independent stream per tensor,
seeded with ``SeedSequence([seed, stream_id])``.  Values are drawn in fp32
(uniform via ``Generator.random``, normal via ``Generator.standard_normal``),
then rounded once to the tensor's storage type.  "N(0, s)" means standard
deviation s; the conv weights of the two large convolutions use variance
1/fan_in, i.e. standard deviation 1/sqrt(fan_in).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bfloat16 (ties to even); return the uint16 words."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact fp32 values of bfloat16 words."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(stream)])))


def _uniform(rng, shape, lo, hi):
    return (lo + (hi - lo) * rng.random(shape, dtype=np.float32)).astype(np.float32)


def _normal(rng, shape, std):
    return (rng.standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


@dataclass(frozen=True)
class ConvShape:
    N: int
    H: int
    W: int
    C_in: int
    C_out: int
    KH: int
    KW: int
    stride: tuple = (1, 1)
    pad: tuple = (0, 0)

    @property
    def Ho(self) -> int:
        return (self.H + 2 * self.pad[0] - self.KH) // self.stride[0] + 1

    @property
    def Wo(self) -> int:
        return (self.W + 2 * self.pad[1] - self.KW) // self.stride[1] + 1

    @property
    def M(self) -> int:
        return self.N * self.Ho * self.Wo

    @property
    def K(self) -> int:
        return self.KH * self.KW * self.C_in

    @property
    def flops(self) -> int:
        return 2 * self.M * self.C_out * self.K


def conv_inputs(shape: ConvShape, seed: int = 0, w_dist: str = "uniform") -> dict:
    """x NHWC bf16 U[-1,1]; w OIHW bf16 (U[-1,1] or N(0, var 1/fan_in));
    bn_scale fp32 U[0.5,1.5]; bn_bias fp32 N(0, 0.1).  Streams 0..3 in that order."""
    s = shape
    x = f32_to_bf16_bits(_uniform(_rng(seed, 0), (s.N, s.H, s.W, s.C_in), -1.0, 1.0))
    wshape = (s.C_out, s.C_in, s.KH, s.KW)
    if w_dist == "uniform":
        w = _uniform(_rng(seed, 1), wshape, -1.0, 1.0)
    elif w_dist == "normal_fanin":
        w = _normal(_rng(seed, 1), wshape, 1.0 / np.sqrt(s.KH * s.KW * s.C_in))
    else:
        raise ValueError(w_dist)
    scale = _uniform(_rng(seed, 2), (s.C_out,), 0.5, 1.5)
    bias = _normal(_rng(seed, 3), (s.C_out,), 0.1)
    return {"x": x, "w_oihw": f32_to_bf16_bits(w), "scale": scale, "bias": bias}


def bias_gelu_inputs(rows: int, cols: int, seed: int = 0) -> dict:
    """x fp16 [rows, cols] N(0,1); bias fp16 [cols] N(0,0.1).  Streams 0, 1."""
    x = _normal(_rng(seed, 0), (rows, cols), 1.0).astype(np.float16)
    bias = _normal(_rng(seed, 1), (cols,), 0.1).astype(np.float16)
    return {"x": x, "bias": bias}


def layernorm_inputs(rows: int, hidden: int, seed: int = 0) -> dict:
    """act, res fp16 [rows, hidden] N(0,1); gamma fp32 U[0.5,1.5]; beta fp32 N(0,0.1).
    Streams 0..3 in that order."""
    act = _normal(_rng(seed, 0), (rows, hidden), 1.0).astype(np.float16)
    res = _normal(_rng(seed, 1), (rows, hidden), 1.0).astype(np.float16)
    gamma = _uniform(_rng(seed, 2), (hidden,), 0.5, 1.5)
    beta = _normal(_rng(seed, 3), (hidden,), 0.1)
    return {"act": act, "res": res, "gamma": gamma, "beta": beta}


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "conv", "bias_gelu", "bias_gelu_rowsum" or "layernorm"
    conv: ConvShape | None = None
    w_dist: str = "uniform"
    rows: int = 0
    cols: int = 0
    eps: float = 1e-5
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("conv3x3_tiny_1x16x16x8_to16", "conv",
                 ConvShape(1, 16, 16, 8, 16, 3, 3, (1, 1), (1, 1)), "uniform"),
        Workload("bias_gelu_f16_8192x8192", "bias_gelu", rows=8192, cols=8192),
        Workload("bias_gelu_rowsum_f16_8192x8192", "bias_gelu_rowsum", rows=8192, cols=8192),
        Workload("residual_layernorm_f16_16384x4096", "layernorm", rows=16384, cols=4096, eps=1e-5),
        Workload("conv1x1_32x56x56x256_to256", "conv",
                 ConvShape(32, 56, 56, 256, 256, 1, 1, (1, 1), (0, 0)), "normal_fanin"),
        Workload("conv7x7_16x64x64x512_to512", "conv",
                 ConvShape(16, 64, 64, 512, 512, 7, 7, (1, 1), (3, 3)), "normal_fanin"),
    ]
}


# Producer -> consumer pair ("When the fusion you want is impossible, fuse into
# the producer"): a pointwise activation between two convolutions, the
# consumer a 7x7 conv.  Producer: 1x1, 256 -> 128 channels; consumer: 7x7,
# 128 -> 128, pad 3, both on 16 x 64 x 64 NHWC bf16.
PAIR_PRODUCER = ConvShape(16, 64, 64, 256, 128, 1, 1, (1, 1), (0, 0))
PAIR_CONSUMER = ConvShape(16, 64, 64, 128, 128, 7, 7, (1, 1), (3, 3))


def producer_consumer_inputs(producer: ConvShape, consumer: ConvShape, seed: int = 0) -> dict:
    """Inputs of both convs: the producer's x, w, scale, bias (streams 0..3)
    and the consumer's w, scale, bias (streams 11..13), weights N(0, var 1/fan_in)."""
    a = conv_inputs(producer, seed, "normal_fanin")
    c = consumer
    w2 = _normal(_rng(seed, 11), (c.C_out, c.C_in, c.KH, c.KW), 1.0 / np.sqrt(c.KH * c.KW * c.C_in))
    return {"x": a["x"], "w1_oihw": a["w_oihw"], "scale1": a["scale"], "bias1": a["bias"],
            "w2_oihw": f32_to_bf16_bits(w2), "scale2": _uniform(_rng(seed, 12), (c.C_out,), 0.5, 1.5),
            "bias2": _normal(_rng(seed, 13), (c.C_out,), 0.1)}


def workload_inputs(w: Workload, seed: int = 0) -> dict:
    if w.kind == "conv":
        return conv_inputs(w.conv, seed, w.w_dist)
    if w.kind in ("bias_gelu", "bias_gelu_rowsum"):
        return bias_gelu_inputs(w.rows, w.cols, seed)
    if w.kind == "layernorm":
        return layernorm_inputs(w.rows, w.cols, seed)
    raise ValueError(w.kind)
