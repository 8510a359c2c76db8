"""GPU parity on seeded random shapes: every conv kernel the shape admits
(and the dispatch's own choice), bias + GELU at random widths on both sides of
the bulk-copy ring's 16384-column limit, and residual LayerNorm at random
widths under every row-reduction strategy that takes the width.  Same
oracle, same tolerances as test_gpu_parity.py."""
import numpy as np
import pytest
import torch

import oracle
from gemm_conv_epilogues_gb300 import synth
from helpers import bf16_to_f64, dev_f16, dev_f32, dev_u16, f16_ulp_distance, host_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def b(cuda_ready):
    from gemm_conv_epilogues_gb300 import binding
    return binding


def _random_convs(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        kh, kw = (int(v) for v in rng.choice([1, 3, 5, 7], 2))
        sh, sw = (int(v) for v in rng.choice([1, 2], 2))
        ph, pw = int(rng.integers(0, kh // 2 + 1)), int(rng.integers(0, kw // 2 + 1))
        N = int(rng.integers(1, 3))
        H, W = int(rng.integers(3, 21)), int(rng.integers(3, 21))
        c_in = int(rng.choice([8, 16, 24, 64, 128]))
        c_out = int(rng.choice([8, 16, 32, 48, 64, 96, 128, 256]))
        c = synth.ConvShape(N, H, W, c_in, c_out, kh, kw, (sh, sw), (ph, pw))
        if c.Ho >= 1 and c.Wo >= 1:
            out.append(c)
    return out


CONVS = _random_convs(24, seed=2024)


@pytest.mark.parametrize("c", CONVS, ids=lambda c: f"{c.N}x{c.H}x{c.W}x{c.C_in}-{c.C_out}k{c.KH}{c.KW}"
                                                   f"s{c.stride[0]}{c.stride[1]}p{c.pad[0]}{c.pad[1]}")
def test_conv_random_shape_every_kernel(b, c):
    d = synth.conv_inputs(c, seed=40, w_dist="normal_fanin")
    ref = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], c.stride, c.pad)
    x = dev_u16(d["x"])
    w = torch.empty((c.C_out, c.KH, c.KW, c.C_in), dtype=torch.int16, device="cuda")
    b.tf_pack_filter_nhwc(dev_u16(d["w_oihw"]), w, c.C_out, c.C_in, c.KH, c.KW)
    sc, bi = dev_f32(d["scale"]), dev_f32(d["bias"])
    shape = b.conv_shape(c.N, c.H, c.W, c.C_in, c.C_out, c.KH, c.KW, c.stride, c.pad)
    # the tensor-core kernel takes every shape here (channel tails included);
    # its paired and wide forms need whole 32- and 256-channel tiles
    variants = [b.TF_CONV_AUTO, b.TF_CONV_DIRECT, b.TF_CONV_TILED, b.TF_CONV_UMMA]
    if c.C_out % 32 == 0:
        variants.append(b.TF_CONV_UMMA_PAIR)
    if c.C_out % 256 == 0:
        variants += [b.TF_CONV_UMMA_PAIR_WIDE, b.TF_CONV_UMMA_WIDE]
    for v in variants:
        y = torch.full((c.M, c.C_out), 0x7FC0, dtype=torch.int16, device="cuda")   # NaN sentinel
        b.tf_conv2d_bn_silu_variant(x, w, sc, bi, y, shape, v)
        torch.cuda.synchronize()
        got = bf16_to_f64(host_u16(y)).reshape(ref.shape)
        err = np.abs(got - ref)
        bad = err > 1e-2 + 1e-2 * np.abs(ref)
        assert not bad.any(), f"variant {v}: {bad.sum()} outside tolerance, worst {err.max():.4g}"
    rc, word = b.tf_read_device_error()
    assert rc == b.TF_OK and word == 0


def _random_widths(n, seed, hi):
    rng = np.random.default_rng(seed)
    return [(int(rng.integers(1, 64)), 8 * int(rng.integers(1, hi // 8 + 1))) for _ in range(n)]


@pytest.mark.parametrize("rows,cols", _random_widths(12, seed=7, hi=24000))
def test_bias_gelu_random_width(b, rows, cols):
    d = synth.bias_gelu_inputs(rows, cols, seed=41)
    y = torch.empty((rows, cols), dtype=torch.float16, device="cuda")
    b.tf_bias_gelu(dev_f16(d["x"]), dev_f16(d["bias"]), y, rows, cols)
    torch.cuda.synchronize()
    ulp = f16_ulp_distance(y.cpu().numpy().view(np.uint16), oracle.bias_gelu(d["x"], d["bias"]))
    assert ulp.max() <= 2


@pytest.mark.parametrize("rows,cols", _random_widths(6, seed=9, hi=16384)
                         + [(r, 256 * (c // 256 + 1)) for r, c in _random_widths(6, seed=10, hi=16000)])
def test_bias_gelu_rowsum_random_width(b, rows, cols):
    # half the widths multiples of 256, half arbitrary multiples of 8
    d = synth.bias_gelu_inputs(rows, cols, seed=43)
    y = torch.empty((rows, cols), dtype=torch.float16, device="cuda")
    rs = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
    b.tf_bias_gelu_rowsum(dev_f16(d["x"]), dev_f16(d["bias"]), y, rs, rows, cols)
    torch.cuda.synchronize()
    ref_y, _ = oracle.bias_gelu_rowsum(d["x"], d["bias"])
    assert f16_ulp_distance(y.cpu().numpy().view(np.uint16), ref_y).max() <= 2
    err = np.abs(rs.cpu().numpy().astype(np.float64) - ref_y.sum(axis=1))
    assert np.all(err <= 1e-3 * np.abs(ref_y).sum(axis=1) + 1e-3)
    rc, word = b.tf_read_device_error()
    assert rc == b.TF_OK and word == 0


@pytest.mark.parametrize("rows,hidden", _random_widths(12, seed=8, hi=48000))
def test_layernorm_random_width_every_strategy(b, rows, hidden):
    d = synth.layernorm_inputs(rows, hidden, seed=42)
    ref = oracle.residual_layernorm(d["act"], d["res"], d["gamma"], d["beta"], eps=1e-5)
    act, res = dev_f16(d["act"]), dev_f16(d["res"])
    g, be = dev_f32(d["gamma"]), dev_f32(d["beta"])
    ran = 0
    for v in (b.TF_LN_AUTO, b.TF_LN_WARP, b.TF_LN_CTA, b.TF_LN_CLUSTER):
        y = torch.full((rows, hidden), float("nan"), dtype=torch.float16, device="cuda")
        rc = b.tf_residual_layernorm_variant(act, res, g, be, y, rows, hidden, 1e-5, v, check=False)
        if rc == b.TF_ERR_UNSUPPORTED:   # the strategy does not take this width
            continue
        assert rc == b.TF_OK, (v, rc)
        torch.cuda.synchronize()
        err = np.abs(y.cpu().numpy().astype(np.float64) - ref)
        assert err.max() <= 1e-2, (v, err.max())
        ran += 1
    assert ran >= 2   # the dispatch's choice and at least that strategy forced
    rc, word = b.tf_read_device_error()
    assert rc == b.TF_OK and word == 0


def test_calls_captured_in_a_cuda_graph(b):
    # conv -> bias+GELU -> LayerNorm captured once (programmatic launches become
    # graph edges) and replayed three times on new inputs; each replay matches
    # the oracle
    c = synth.ConvShape(2, 16, 16, 64, 128, 3, 3, (1, 1), (1, 1))
    w = torch.empty((c.C_out, c.KH, c.KW, c.C_in), dtype=torch.int16, device="cuda")
    d0 = synth.conv_inputs(c, seed=50, w_dist="normal_fanin")
    b.tf_pack_filter_nhwc(dev_u16(d0["w_oihw"]), w, c.C_out, c.C_in, c.KH, c.KW)
    sc, bi = dev_f32(d0["scale"]), dev_f32(d0["bias"])
    shape = b.conv_shape(c.N, c.H, c.W, c.C_in, c.C_out, c.KH, c.KW, c.stride, c.pad)
    rows, cols = 64, 4096
    x = torch.empty((c.N, c.H, c.W, c.C_in), dtype=torch.int16, device="cuda")
    y = torch.empty((c.M, c.C_out), dtype=torch.int16, device="cuda")
    g_in = torch.empty((rows, cols), dtype=torch.float16, device="cuda")
    g_bias = torch.empty((cols,), dtype=torch.float16, device="cuda")
    g_out = torch.empty_like(g_in)
    res = torch.empty_like(g_in)
    gam = torch.empty((cols,), dtype=torch.float32, device="cuda")
    bet = torch.empty_like(gam)
    ln_out = torch.empty_like(g_in)
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        s = torch.cuda.current_stream()
        b.tf_conv2d_bn_silu(x, w, sc, bi, y, shape, stream=s)
        b.tf_bias_gelu(g_in, g_bias, g_out, rows, cols, stream=s)
        b.tf_residual_layernorm(g_out, res, gam, bet, ln_out, rows, cols, 1e-5, stream=s)
    for k in range(3):
        d = synth.conv_inputs(c, seed=51 + k, w_dist="normal_fanin")
        e = synth.bias_gelu_inputs(rows, cols, seed=61 + k)
        f = synth.layernorm_inputs(rows, cols, seed=71 + k)
        x.copy_(dev_u16(d["x"]))
        g_in.copy_(dev_f16(e["x"]))
        g_bias.copy_(dev_f16(e["bias"]))
        res.copy_(dev_f16(f["res"]))
        gam.copy_(dev_f32(f["gamma"]))
        bet.copy_(dev_f32(f["beta"]))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        ref = oracle.conv2d_bn_silu(d["x"], d0["w_oihw"], d0["scale"], d0["bias"], c.stride, c.pad)
        got = bf16_to_f64(host_u16(y)).reshape(ref.shape)
        assert np.all(np.abs(got - ref) <= 1e-2 + 1e-2 * np.abs(ref))
        assert f16_ulp_distance(g_out.cpu().numpy().view(np.uint16), oracle.bias_gelu(e["x"], e["bias"])).max() <= 2
        ref_ln = oracle.residual_layernorm(g_out.cpu().numpy(), f["res"], f["gamma"], f["beta"], eps=1e-5)
        assert np.abs(ln_out.cpu().numpy().astype(np.float64) - ref_ln).max() <= 1e-2
    rc, word = b.tf_read_device_error()
    assert rc == b.TF_OK and word == 0


@pytest.mark.parametrize("variant", ["pair", "wide", "wide_tail_launch"])
def test_cluster_conv_captured_in_a_cuda_graph(b, variant):
    # the CTA-pair kernels (cluster and programmatic-launch attributes)
    # captured once and replayed on new inputs: wide tiles with their
    # half-tile tail, and a full wave of wide tiles whose partial last wave
    # is a second launch (two kernels in the graph)
    v = b.TF_CONV_UMMA_PAIR if variant == "pair" else b.TF_CONV_UMMA_PAIR_WIDE
    c = synth.ConvShape(2, 20, 20, 64, 256, 3, 3, (1, 1), (1, 1))
    if variant == "wide_tail_launch":
        c = synth.ConvShape(11, 61, 61, 64, 256, 3, 3, (1, 1), (1, 1))
    d0 = synth.conv_inputs(c, seed=80, w_dist="normal_fanin")
    w = torch.empty((c.C_out, c.KH, c.KW, c.C_in), dtype=torch.int16, device="cuda")
    b.tf_pack_filter_nhwc(dev_u16(d0["w_oihw"]), w, c.C_out, c.C_in, c.KH, c.KW)
    sc, bi = dev_f32(d0["scale"]), dev_f32(d0["bias"])
    shape = b.conv_shape(c.N, c.H, c.W, c.C_in, c.C_out, c.KH, c.KW, c.stride, c.pad)
    x = torch.empty((c.N, c.H, c.W, c.C_in), dtype=torch.int16, device="cuda")
    y = torch.empty((c.M, c.C_out), dtype=torch.int16, device="cuda")
    x.copy_(dev_u16(d0["x"]))
    b.tf_conv2d_bn_silu_variant(x, w, sc, bi, y, shape, v)   # first call outside the capture
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        b.tf_conv2d_bn_silu_variant(x, w, sc, bi, y, shape, v, stream=torch.cuda.current_stream())
    for k in range(3):
        d = synth.conv_inputs(c, seed=81 + k, w_dist="normal_fanin")
        x.copy_(dev_u16(d["x"]))
        y.fill_(0x7FC0)   # NaN sentinel: every output must be rewritten by the replay
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        ref = oracle.conv2d_bn_silu(d["x"], d0["w_oihw"], d0["scale"], d0["bias"], c.stride, c.pad)
        got = bf16_to_f64(host_u16(y)).reshape(ref.shape)
        assert np.all(np.abs(got - ref) <= 1e-2 + 1e-2 * np.abs(ref))
    rc, word = b.tf_read_device_error()
    assert rc == b.TF_OK and word == 0

