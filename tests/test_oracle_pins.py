"""Pins for the CPU oracle, each against something other than the oracle itself:
library routines (numpy's IEEE fp16 conversion, torch's fp64 conv2d and
layer_norm, scipy's correlate2d and ndtr), printed tables (tests/golden/) and
closed forms.  No GPU involved."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from gemm_conv_epilogues_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _table(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append([float(t) for t in line.split()])
    return np.array(rows)


# ---------------------------------------------------------------- formats

def test_f16_decode_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_value(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def test_bf16_decode_matches_torch():
    bits = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = np.array([oracle.bf16_value(int(b)) for b in bits])
    ok = np.isfinite(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_round_to_f16_matches_numpy_ieee_rounding():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 5, 4000),
        # exact ties between adjacent fp16 values (normal and subnormal)
        (np.arange(1, 300, dtype=np.float64) + 0.5) * 2.0 ** -24,
        (np.arange(1024, 1400, dtype=np.float64) + 0.5) * 2.0 ** -10,
        np.array([65504.0, 65519.9, 65520.0, -65520.0, 0.0, -0.0, 6e-8, 2.9e-8, 3.0e-8]),
    ])
    ref = vals.astype(np.float16).astype(np.float64)
    got = np.array([oracle.round_to_f16(float(v)) for v in vals])
    assert np.array_equal(got, ref)


def test_round_to_bf16_matches_torch_on_fp32_values():
    rng = np.random.default_rng(2)
    vals = (rng.standard_normal(5000) * 10.0 ** rng.integers(-30, 30, 5000)).astype(np.float32)
    ties = ((np.arange(128, 256, dtype=np.float32) + 0.5) * np.float32(2.0 ** -3)).astype(np.float32)
    vals = np.concatenate([vals, ties, -ties])
    ref = torch.from_numpy(vals).to(torch.bfloat16).double().numpy()
    got = np.array([oracle.round_to_bf16(float(v)) for v in vals])
    assert np.array_equal(got, ref)


def test_synth_bf16_rounding_agrees_with_torch():
    rng = np.random.default_rng(3)
    vals = rng.standard_normal(20000).astype(np.float32)
    mine = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(vals))
    ref = torch.from_numpy(vals).to(torch.bfloat16).float().numpy()
    assert np.array_equal(mine, ref)


# ---------------------------------------------------------------- SiLU / GELU

def test_silu_against_logistic_table():
    for v, sig in _table("logistic.txt"):
        assert abs(oracle.silu(v) - v * sig) <= 1e-12 * max(1.0, abs(v))
    assert oracle.silu(0.0) == 0.0


def test_gelu_against_normal_table():
    for z, phi in _table("normal_cdf.txt"):
        ref = z * phi
        assert abs(oracle.gelu(z) - ref) <= 1e-10 * abs(ref) + 1e-300, (z, oracle.gelu(z), ref)


def test_gelu_closed_forms():
    from scipy.special import ndtr
    assert oracle.gelu(0.0) == 0.0
    rng = np.random.default_rng(4)
    for s in rng.uniform(-8, 8, 400):
        # Phi(-s) = 1 - Phi(s)  =>  GELU(-s) = GELU(s) - s
        assert abs(oracle.gelu(-s) - (oracle.gelu(s) - s)) <= 1e-12 * max(1.0, abs(s))
        ref = s * ndtr(s)
        assert abs(oracle.gelu(s) - ref) <= 1e-13 * max(abs(ref), 1e-300) + 1e-300
    for s in (7.5, 9.0, 12.0):
        assert abs(oracle.gelu(s) - s) < 1e-10
    # deep negative tail keeps relative accuracy (no 1 + erf cancellation)
    assert abs(oracle.gelu(-7.0) / (-7.0 * ndtr(-7.0)) - 1.0) < 1e-12


def test_bias_gelu_broadcasts_bias_over_columns():
    rows, cols = 3, 40
    x = np.zeros((rows, cols), np.float16)
    bias = np.linspace(-3, 3, cols).astype(np.float16)
    y = oracle.bias_gelu(x, bias)
    expect = np.array([oracle.gelu(float(b)) for b in bias.astype(np.float64)])
    for r in range(rows):
        assert np.array_equal(y[r], expect)
    # a column-constant input shifted by a row-constant bias would differ: rows are not biased
    x2 = np.tile(np.arange(rows, dtype=np.float16)[:, None], (1, cols))
    y2 = oracle.bias_gelu(x2, np.zeros(cols, np.float16))
    assert np.allclose(y2[:, 0], [oracle.gelu(float(r)) for r in range(rows)], rtol=0, atol=0)


def test_bias_gelu_matches_scipy_ndtr():
    from scipy.special import ndtr
    d = synth.bias_gelu_inputs(64, 96, seed=5)
    y = oracle.bias_gelu(d["x"], d["bias"])
    s = d["x"].astype(np.float64) + d["bias"].astype(np.float64)[None, :]
    ref = s * ndtr(s)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-300)


def test_bias_gelu_materialized_sum_is_rounded_to_f16():
    d = synth.bias_gelu_inputs(16, 64, seed=6)
    y_chain = oracle.bias_gelu(d["x"], d["bias"], materialize=True)
    s16 = (d["x"].astype(np.float64) + d["bias"].astype(np.float64)[None, :]).astype(np.float16)
    y_from_s16 = oracle.bias_gelu(s16, np.zeros(64, np.float16))
    assert np.array_equal(y_chain, y_from_s16)


def test_bias_gelu_rowsum_is_row_sum():
    d = synth.bias_gelu_inputs(32, 80, seed=7)
    y, rs = oracle.bias_gelu_rowsum(d["x"], d["bias"])
    assert np.array_equal(y, oracle.bias_gelu(d["x"], d["bias"]))
    assert np.allclose(rs, y.sum(axis=1), rtol=1e-13, atol=1e-12)


# ---------------------------------------------------------------- conv

def _torch_conv(x_bits, w_bits, scale, bias, stride, pad, epilogue):
    x = torch.from_numpy(synth.bf16_bits_to_f32(x_bits).astype(np.float64)).permute(0, 3, 1, 2)
    w = torch.from_numpy(synth.bf16_bits_to_f32(w_bits).astype(np.float64))
    acc = torch.nn.functional.conv2d(x, w, stride=stride, padding=pad).permute(0, 2, 3, 1).numpy()
    if epilogue == oracle.EPI_NONE:
        return acc
    v = acc * scale.astype(np.float64) + bias.astype(np.float64)
    return v / (1.0 + np.exp(-v))


@pytest.mark.parametrize("shape", [
    synth.ConvShape(1, 5, 6, 2, 3, 3, 3, (1, 1), (1, 1)),
    synth.ConvShape(2, 7, 5, 3, 4, 3, 2, (2, 1), (1, 0)),
    synth.ConvShape(1, 9, 9, 4, 2, 7, 7, (1, 1), (3, 3)),
    synth.ConvShape(2, 6, 6, 5, 3, 1, 1, (2, 2), (0, 0)),
    synth.ConvShape(1, 8, 8, 3, 2, 5, 3, (3, 2), (2, 1)),
])
def test_conv_matches_torch_fp64(shape):
    d = synth.conv_inputs(shape, seed=8)
    for epi in (oracle.EPI_NONE, oracle.EPI_FUSED):
        y = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], shape.stride, shape.pad, epi)
        ref = _torch_conv(d["x"], d["w_oihw"], d["scale"], d["bias"], shape.stride, shape.pad, epi)
        assert y.shape == (shape.N, shape.Ho, shape.Wo, shape.C_out)
        assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_conv_matches_scipy_correlate2d():
    from scipy.signal import correlate2d
    shape = synth.ConvShape(1, 6, 7, 2, 2, 3, 3, (1, 1), (1, 1))
    d = synth.conv_inputs(shape, seed=9)
    y = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], (1, 1), (1, 1), oracle.EPI_NONE)
    x = synth.bf16_bits_to_f32(d["x"]).astype(np.float64)[0]
    w = synth.bf16_bits_to_f32(d["w_oihw"]).astype(np.float64)
    for co in range(2):
        ref = sum(correlate2d(x[:, :, ci], w[co, ci], mode="same", boundary="fill") for ci in range(2))
        assert np.allclose(y[0, :, :, co], ref, rtol=1e-12, atol=1e-12)


def test_conv1x1_is_a_matmul():
    shape = synth.ConvShape(2, 4, 3, 16, 8, 1, 1)
    d = synth.conv_inputs(shape, seed=10)
    y = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], epilogue=oracle.EPI_NONE)
    a = synth.bf16_bits_to_f32(d["x"]).astype(np.float64).reshape(-1, 16)
    b = synth.bf16_bits_to_f32(d["w_oihw"]).astype(np.float64).reshape(8, 16)
    assert np.allclose(y.reshape(-1, 8), a @ b.T, rtol=1e-12, atol=1e-12)


def test_conv_all_ones_closed_form():
    # x = 1, w = 1, 3x3, pad 1: each output sums the in-bounds taps, 9*C_in
    # inside, 6*C_in on edges, 4*C_in at corners; scale 1, bias 0 -> SiLU of that.
    n, h, w, ci, co = 1, 5, 4, 3, 2
    one = synth.f32_to_bf16_bits(np.ones(1, np.float32))[0]
    x = np.full((n, h, w, ci), one, np.uint16)
    wt = np.full((co, ci, 3, 3), one, np.uint16)
    y = oracle.conv2d_bn_silu(x, wt, np.ones(co, np.float32), np.zeros(co, np.float32), (1, 1), (1, 1))
    for i in range(h):
        for j in range(w):
            taps = (3 - (i == 0) - (i == h - 1)) * (3 - (j == 0) - (j == w - 1))
            a = taps * ci
            assert np.allclose(y[0, i, j], a / (1 + math.exp(-a)), rtol=1e-15)


def test_conv_zero_input_gives_silu_of_bias():
    shape = synth.ConvShape(1, 5, 5, 4, 6, 3, 3, (1, 1), (1, 1))
    d = synth.conv_inputs(shape, seed=11)
    x0 = np.zeros_like(d["x"])
    y = oracle.conv2d_bn_silu(x0, d["w_oihw"], d["scale"], d["bias"], (1, 1), (1, 1))
    for co in range(6):
        assert np.all(y[..., co] == oracle.silu(float(d["bias"][co])))
    y0 = oracle.conv2d_bn_silu(x0, d["w_oihw"], d["scale"], np.zeros(6, np.float32), (1, 1), (1, 1))
    assert np.all(y0 == 0.0)


def test_conv_unit_scale_zero_bias_is_conv_then_silu():
    shape = synth.ConvShape(1, 6, 6, 3, 4, 3, 3, (1, 1), (1, 1))
    d = synth.conv_inputs(shape, seed=12)
    acc = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], (1, 1), (1, 1), oracle.EPI_NONE)
    y = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], np.ones(4, np.float32), np.zeros(4, np.float32), (1, 1), (1, 1))
    from scipy.special import expit
    assert np.allclose(y, acc * expit(acc), rtol=1e-13, atol=1e-15)


def test_conv_points_equal_full_output():
    shape = synth.ConvShape(2, 7, 6, 3, 5, 3, 3, (2, 1), (1, 1))
    d = synth.conv_inputs(shape, seed=13)
    y = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], shape.stride, shape.pad)
    pts = np.random.default_rng(0).integers(0, y.size, 50)
    yp = oracle.conv2d_bn_silu_points(d["x"], d["w_oihw"], d["scale"], d["bias"], pts, shape.stride, shape.pad)
    assert np.array_equal(yp, y.reshape(-1)[pts])


def test_conv_chain_rounds_only_at_the_boundaries():
    # integer data: acc and acc*1+0 are exact in bf16 -> chain == fused
    rng = np.random.default_rng(14)
    x = synth.f32_to_bf16_bits(rng.integers(-2, 3, (1, 4, 4, 2)).astype(np.float32))
    w = synth.f32_to_bf16_bits(rng.integers(-2, 3, (3, 2, 3, 3)).astype(np.float32))
    ones, zeros = np.ones(3, np.float32), np.zeros(3, np.float32)
    a = oracle.conv2d_bn_silu(x, w, ones, zeros, (1, 1), (1, 1), oracle.EPI_FUSED)
    b = oracle.conv2d_bn_silu(x, w, ones, zeros, (1, 1), (1, 1), oracle.EPI_CHAIN)
    assert np.array_equal(a, b)
    # random data: the chain stays within two bf16 roundings of the fused value
    shape = synth.ConvShape(1, 6, 6, 8, 4, 3, 3, (1, 1), (1, 1))
    d = synth.conv_inputs(shape, seed=15)
    f = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], (1, 1), (1, 1), oracle.EPI_FUSED)
    c = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], (1, 1), (1, 1), oracle.EPI_CHAIN)
    acc = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], (1, 1), (1, 1), oracle.EPI_NONE)
    bound = 2 * 2.0 ** -8 * (np.abs(acc) * d["scale"].max() + 1.0) * 1.2
    assert np.all(np.abs(f - c) <= bound)
    assert np.any(f != c)


# ---------------------------------------------------------------- pack

def test_pack_filter_is_the_ohwi_permutation():
    rng = np.random.default_rng(16)
    w = rng.integers(0, 65536, (5, 3, 7, 2)).astype(np.uint16)
    p = oracle.pack_filter(w)
    assert np.array_equal(p, np.transpose(w, (0, 2, 3, 1)))
    assert np.array_equal(np.transpose(p, (0, 3, 1, 2)), w)           # unpack . pack = id
    w1 = rng.integers(0, 65536, (4, 6, 1, 1)).astype(np.uint16)
    assert np.array_equal(oracle.pack_filter(w1).reshape(-1), w1.reshape(-1))   # 1x1: identity


# ---------------------------------------------------------------- LayerNorm

def test_layernorm_hand_rows():
    t = _table("layernorm_rows.txt")
    act = t[:, 0:4].astype(np.float16)
    res = t[:, 4:8].astype(np.float16)
    y = oracle.residual_layernorm(act, res, np.ones(4, np.float32), np.zeros(4, np.float32), eps=0.0)
    assert np.allclose(y, t[:, 8:12], rtol=0, atol=1e-15)


def test_layernorm_matches_torch_fp64():
    d = synth.layernorm_inputs(24, 200, seed=17)
    y, st = oracle.residual_layernorm(d["act"], d["res"], d["gamma"], d["beta"], eps=1e-5, want_stats=True)
    s = torch.from_numpy(d["act"].astype(np.float64) + d["res"].astype(np.float64))
    ref = torch.nn.functional.layer_norm(s, (200,), torch.from_numpy(d["gamma"].astype(np.float64)),
                                         torch.from_numpy(d["beta"].astype(np.float64)), eps=1e-5).numpy()
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    sn = s.numpy()
    assert np.allclose(st[:, 0], sn.mean(axis=1), rtol=0, atol=1e-13)
    assert np.allclose(st[:, 1], sn.var(axis=1), rtol=1e-12, atol=0)


def test_layernorm_rows_are_standardised_before_affine():
    d = synth.layernorm_inputs(16, 512, seed=18)
    y, st = oracle.residual_layernorm(d["act"], d["res"], np.ones(512, np.float32),
                                      np.zeros(512, np.float32), eps=1e-5, want_stats=True)
    assert np.all(np.abs(y.mean(axis=1)) < 1e-12)
    assert np.allclose(y.var(axis=1), st[:, 1] / (st[:, 1] + 1e-5), rtol=1e-12)


def test_layernorm_shift_invariance_and_affine():
    d = synth.layernorm_inputs(8, 64, seed=19)
    g1, b0 = np.ones(64, np.float32), np.zeros(64, np.float32)
    base = oracle.residual_layernorm(d["act"], d["res"], g1, b0)
    shifted = oracle.residual_layernorm(d["act"], (d["res"].astype(np.float32) + 4.0).astype(np.float16), g1, b0)
    # adding 4 to an fp16 value can round; compare on rows where the shift stayed exact
    exact = np.all(shifted.shape == base.shape)
    assert exact
    s0 = d["act"].astype(np.float64) + d["res"].astype(np.float64)
    s1 = d["act"].astype(np.float64) + (d["res"].astype(np.float32) + 4.0).astype(np.float16).astype(np.float64)
    ok = np.all(np.abs((s1 - s0) - 4.0) == 0.0, axis=1)
    assert np.allclose(shifted[ok], base[ok], rtol=0, atol=1e-12)
    y = oracle.residual_layernorm(d["act"], d["res"], d["gamma"], d["beta"])
    assert np.allclose(y, base * d["gamma"].astype(np.float64) + d["beta"].astype(np.float64), rtol=1e-15, atol=1e-15)


def test_layernorm_materialized_chain():
    d = synth.layernorm_inputs(8, 128, seed=20)
    y = oracle.residual_layernorm(d["act"], d["res"], d["gamma"], d["beta"], materialize=True)
    s16 = (d["act"].astype(np.float64) + d["res"].astype(np.float64)).astype(np.float16)
    n = oracle.residual_layernorm(s16, np.zeros_like(s16), np.ones(128, np.float32), np.zeros(128, np.float32))
    ref = n.astype(np.float16).astype(np.float64) * d["gamma"].astype(np.float64) + d["beta"].astype(np.float64)
    assert np.allclose(y, ref, rtol=0, atol=1e-15)


def test_conv_chain_matches_library_rounded_boundaries():
    # t1 = bf16(acc), t2 = bf16(t1*scale + bias), y = SiLU(t2), with the roundings
    # done by torch's bfloat16 conversion instead of the oracle's own.
    from scipy.special import expit
    shape = synth.ConvShape(1, 8, 8, 16, 8, 3, 3, (1, 1), (1, 1))
    d = synth.conv_inputs(shape, seed=21)
    acc = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], (1, 1), (1, 1), oracle.EPI_NONE)
    r = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).double().numpy()
    t1 = r(acc)
    t2 = r(t1 * d["scale"].astype(np.float64) + d["bias"].astype(np.float64))
    ref = t2 * expit(t2)
    c = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], (1, 1), (1, 1), oracle.EPI_CHAIN)
    assert np.allclose(c, ref, rtol=1e-14, atol=1e-300)
