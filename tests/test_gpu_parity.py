"""GPU parity: every kernel behind the C ABI against the fp64 oracle on the
same seeded input bits.

Tolerances:
  conv (bf16 out)       |gpu - ref| <= 1e-2 + 1e-2*|ref|
  bias + GELU (fp16)    <= 2 fp16 ulp from the oracle rounded to fp16
  LayerNorm (fp16)      |gpu - ref| <= 1e-2
  filter pack           bit-identical
"""
import numpy as np
import pytest
import torch

import oracle
from gemm_conv_epilogues_gb300 import synth
from helpers import (bf16_to_f64, conv_sample_points, dev_f16, dev_f32, dev_u16, f16_ulp_distance,
                     host_u16)

pytestmark = pytest.mark.gpu

CONV_ATOL, CONV_RTOL = 1e-2, 1e-2


@pytest.fixture(scope="module")
def b(cuda_ready):
    from gemm_conv_epilogues_gb300 import binding
    return binding


def _shape(b, c):
    return b.conv_shape(c.N, c.H, c.W, c.C_in, c.C_out, c.KH, c.KW, c.stride, c.pad)


def _assert_no_device_error(b):
    rc, word = b.tf_read_device_error()
    assert rc == b.TF_OK and word == 0, (rc, hex(word))


def _conv_check(got, ref):
    err = np.abs(got - ref)
    bound = CONV_ATOL + CONV_RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside tolerance; worst {err.max():.4g}"


def _run_conv(b, c, d, variant, fused=True):
    x = dev_u16(d["x"])
    w = torch.empty((c.C_out, c.KH, c.KW, c.C_in), dtype=torch.int16, device="cuda")
    b.tf_pack_filter_nhwc(dev_u16(d["w_oihw"]), w, c.C_out, c.C_in, c.KH, c.KW)
    y = torch.full((c.N, c.Ho, c.Wo, c.C_out), 0x7FC0, dtype=torch.int16, device="cuda")  # NaN sentinel
    if fused:
        b.tf_conv2d_bn_silu_variant(x, w, dev_f32(d["scale"]), dev_f32(d["bias"]), y, _shape(b, c), variant)
    else:
        b.tf_unfused_conv2d(x, w, y, _shape(b, c), variant)
    torch.cuda.synchronize()
    return bf16_to_f64(host_u16(y))


# ---------------------------------------------------------------- filter pack

@pytest.mark.parametrize("dims", [(16, 8, 3, 3), (256, 256, 1, 1), (64, 24, 7, 7), (5, 3, 2, 4), (1, 1, 1, 1)])
def test_pack_filter_bit_identical(b, dims):
    co, ci, kh, kw = dims
    rng = np.random.default_rng(sum(dims))
    w = rng.integers(0, 65536, dims).astype(np.uint16)
    out = torch.zeros((co, kh, kw, ci), dtype=torch.int16, device="cuda")
    b.tf_pack_filter_nhwc(dev_u16(w), out, co, ci, kh, kw)
    torch.cuda.synchronize()
    assert np.array_equal(host_u16(out), oracle.pack_filter(w))


def test_pack_filter_full_7x7(b):
    d = synth.workload_inputs(synth.WORKLOADS["conv7x7_16x64x64x512_to512"])
    out = torch.zeros((512, 7, 7, 512), dtype=torch.int16, device="cuda")
    b.tf_pack_filter_nhwc(dev_u16(d["w_oihw"]), out, 512, 512, 7, 7)
    torch.cuda.synchronize()
    assert np.array_equal(host_u16(out), oracle.pack_filter(d["w_oihw"]))


# ---------------------------------------------------------------- conv, small shapes, full output

CUDA_CORE_SHAPES = [
    synth.ConvShape(1, 16, 16, 8, 16, 3, 3, (1, 1), (1, 1)),     # the tiny workload
    synth.ConvShape(2, 9, 7, 16, 20, 3, 3, (1, 1), (1, 1)),      # ragged tiles and channel group
    synth.ConvShape(1, 11, 13, 24, 5, 5, 3, (2, 1), (2, 1)),     # stride, non-square kernel and pads
    synth.ConvShape(3, 6, 6, 8, 33, 1, 1, (1, 1), (0, 0)),
    synth.ConvShape(1, 20, 20, 8, 16, 7, 7, (1, 1), (3, 3)),
    # the direct kernel's batched form: a last batch of 7 of 25 units (5x5, 8
    # channels), 45 units over 40 channels at stride 2, and both sides of its
    # 128K-output bound (4x32x32x24 -> 16 batched, -> 32 tap by tap)
    synth.ConvShape(1, 12, 12, 8, 16, 5, 5, (1, 1), (2, 2)),
    synth.ConvShape(2, 16, 16, 40, 24, 3, 3, (2, 2), (1, 1)),
    synth.ConvShape(4, 32, 32, 24, 16, 3, 3, (1, 1), (1, 1)),
    synth.ConvShape(4, 32, 32, 24, 32, 3, 3, (1, 1), (1, 1)),
]


@pytest.mark.parametrize("variant", [0, 1])
@pytest.mark.parametrize("c", CUDA_CORE_SHAPES, ids=lambda c: f"{c.N}x{c.H}x{c.W}x{c.C_in}-{c.C_out}k{c.KH}{c.KW}s{c.stride[0]}{c.stride[1]}")
def test_conv_cuda_core_variants(b, c, variant):
    d = synth.conv_inputs(c, seed=1)
    got = _run_conv(b, c, d, variant)
    ref = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], c.stride, c.pad)
    _conv_check(got, ref)


UMMA_SHAPES = [
    synth.ConvShape(1, 20, 20, 64, 32, 1, 1, (1, 1), (0, 0), ),     # 1x1, one ragged M tile, BN=32
    synth.ConvShape(2, 15, 17, 128, 256, 1, 1, (1, 1), (0, 0)),     # 1x1, several tiles, ragged tail, BN=256
    synth.ConvShape(2, 12, 12, 64, 64, 3, 3, (1, 1), (1, 1)),       # im2col 3x3, tiles cross rows and images
    synth.ConvShape(1, 16, 16, 64, 128, 7, 7, (1, 1), (3, 3)),      # im2col 7x7 pad 3
    synth.ConvShape(2, 10, 14, 128, 96, 3, 3, (1, 1), (1, 1)),      # non-square image, BN=32, 3 N tiles
    synth.ConvShape(1, 17, 17, 64, 64, 3, 3, (2, 2), (1, 1)),       # stride 2
    synth.ConvShape(1, 9, 9, 192, 512, 3, 3, (1, 1), (0, 0)),       # no padding, 2 N tiles of 256
    synth.ConvShape(1, 12, 15, 64, 64, 3, 5, (1, 1), (1, 2)),       # non-square kernel and padding
    synth.ConvShape(2, 10, 10, 64, 64, 1, 7, (1, 1), (0, 3)),       # 1x7
    synth.ConvShape(1, 14, 9, 64, 32, 7, 1, (1, 1), (3, 0)),        # 7x1
    synth.ConvShape(1, 16, 17, 64, 64, 3, 3, (2, 1), (1, 1)),       # different strides along H and W
    synth.ConvShape(1, 17, 16, 64, 64, 3, 3, (2, 2), (1, 1)),       # stride 2 on odd and even extents
    synth.ConvShape(1, 12, 12, 64, 64, 3, 3, (1, 1), (0, 1)),       # padding along W only
    synth.ConvShape(4, 7, 7, 64, 64, 7, 7, (1, 1), (0, 0)),         # 1x1 output: every tap interior
    synth.ConvShape(1, 3, 3, 64, 64, 3, 3, (1, 1), (1, 1)),         # most taps in the padding
    # filter block resident in shared memory (one K split, no pair)
    synth.ConvShape(1, 23, 29, 256, 512, 1, 1, (1, 1), (0, 0)),     # 128 KB block, 2 channel tiles, one tile per CTA
    synth.ConvShape(4, 56, 57, 64, 512, 1, 1, (1, 1), (0, 0)),      # 2 channel tiles, several tiles per CTA
    synth.ConvShape(4, 41, 41, 64, 96, 3, 3, (1, 1), (1, 1)),       # 3 channel tiles of 32, several tiles per CTA
    synth.ConvShape(1, 12, 12, 64, 256, 3, 3, (1, 1), (1, 1)),      # short K, block too big: 128-wide tiles, streamed
    synth.ConvShape(1, 15, 20, 64, 64, 1, 1, (1, 1), (0, 0)),       # plain GEMM, 3 tiles: a pair's second tile wholly past M
    # resident block, one channel tile, more tiles than CTAs: dynamic schedule, half-tile tail
    synth.ConvShape(8, 56, 56, 64, 256, 1, 1, (1, 1), (0, 0)),
]


@pytest.mark.parametrize("variant", [2, 3], ids=["cta", "pair"])
@pytest.mark.parametrize("c", UMMA_SHAPES, ids=lambda c: f"{c.N}x{c.H}x{c.W}x{c.C_in}-{c.C_out}k{c.KH}s{c.stride[0]}p{c.pad[0]}")
def test_conv_umma_small(b, c, variant):
    d = synth.conv_inputs(c, seed=2, w_dist="normal_fanin")
    got = _run_conv(b, c, d, variant)
    ref = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], c.stride, c.pad)
    _conv_check(got, ref)
    _assert_no_device_error(b)


# Channel tails on the tensor-core kernel: C_in not a multiple of 64 (the last
# 64-channel block of each tap zero-filled by TMA, in the filters through
# their 3-D tensor map) and C_out not a multiple of 32 (the last channel
# tile's filter rows zero-filled, its scale/bias masked, its stores clipped;
# C_out % 8 != 0 stores rows that TMA cannot address with masked plain
# stores).  Every output against the oracle.
TAIL_SHAPES = [
    synth.ConvShape(4, 32, 32, 256, 16, 3, 3, (1, 1), (1, 1)),      # C_out 16: one half-empty 32-channel tile
    synth.ConvShape(2, 17, 19, 64, 20, 3, 3, (1, 1), (1, 1)),       # C_out 20: direct stores, ragged M
    synth.ConvShape(2, 20, 20, 128, 48, 3, 3, (2, 2), (1, 1)),      # C_out 48 in a 64 tile, stride 2
    synth.ConvShape(1, 23, 21, 64, 200, 1, 1, (1, 1), (0, 0)),      # C_out 200 in a 256 tile, resident filters
    synth.ConvShape(2, 16, 16, 8, 32, 3, 3, (1, 1), (1, 1)),        # C_in 8: 8 of 64 channels per K step
    synth.ConvShape(1, 18, 18, 24, 64, 5, 5, (1, 1), (2, 2)),       # C_in 24
    synth.ConvShape(3, 11, 13, 40, 96, 1, 1, (1, 1), (0, 0)),       # C_in 40, plain GEMM, 3 tiles of 32
    synth.ConvShape(1, 16, 16, 8, 16, 3, 3, (1, 1), (1, 1)),        # both tails, tiny
    synth.ConvShape(2, 14, 14, 40, 20, 7, 7, (1, 1), (3, 3)),       # both tails, 7x7, direct stores
    synth.ConvShape(1, 20, 20, 72, 300, 3, 3, (1, 1), (1, 1)),      # C_in 64 + 8; C_out 300 = 256 + 44
    synth.ConvShape(2, 9, 9, 136, 5, 1, 1, (1, 1), (0, 0)),         # odd C_out 5: 2-byte rows
]


@pytest.mark.parametrize("c", TAIL_SHAPES, ids=lambda c: f"{c.N}x{c.H}x{c.W}x{c.C_in}-{c.C_out}k{c.KH}s{c.stride[0]}")
def test_conv_umma_channel_tails(b, c):
    d = synth.conv_inputs(c, seed=18, w_dist="normal_fanin")
    got = _run_conv(b, c, d, b.TF_CONV_UMMA)
    ref = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], c.stride, c.pad)
    _conv_check(got, ref)
    _assert_no_device_error(b)


# C_in tails on the paired and wide-tile kernels (which need whole channel tiles)
@pytest.mark.parametrize("variant,c", [
    (3, synth.ConvShape(2, 16, 16, 24, 64, 3, 3, (1, 1), (1, 1))),
    (3, synth.ConvShape(1, 30, 30, 40, 256, 1, 1, (1, 1), (0, 0))),    # paired MMA, resident halves, tail parts
    (4, synth.ConvShape(2, 20, 20, 40, 256, 3, 3, (1, 1), (1, 1))),
    (5, synth.ConvShape(1, 24, 24, 72, 256, 3, 3, (1, 1), (1, 1))),
], ids=["pair-cin24", "pair-1x1-cin40", "pairwide-cin40", "wide-cin72"])
def test_conv_umma_input_channel_tails_other_kernels(b, variant, c):
    d = synth.conv_inputs(c, seed=19, w_dist="normal_fanin")
    got = _run_conv(b, c, d, variant)
    ref = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], c.stride, c.pad)
    _conv_check(got, ref)
    _assert_no_device_error(b)


def test_conv_umma_pair_rejects_channel_tails(b):
    c = synth.ConvShape(1, 12, 12, 64, 48, 3, 3, (1, 1), (1, 1))
    x = torch.zeros((c.N, c.H, c.W, c.C_in), dtype=torch.int16, device="cuda")
    w = torch.zeros((c.C_out, c.KH, c.KW, c.C_in), dtype=torch.int16, device="cuda")
    sc = torch.ones((c.C_out,), dtype=torch.float32, device="cuda")
    y = torch.zeros((c.M, c.C_out), dtype=torch.int16, device="cuda")
    rc = b.tf_conv2d_bn_silu_variant(x, w, sc, sc, y, _shape(b, c), b.TF_CONV_UMMA_PAIR, check=False)
    assert rc == b.TF_ERR_UNSUPPORTED


# 256-pixel tiles per CTA on CTA pairs (C_out % 256 == 0).  With fewer tiles
# than pairs every tile runs as its two 128-row halves (the tail split); the
# second CTA's halves of a pair can lie past M.
WIDE_SHAPES = [
    synth.ConvShape(1, 20, 20, 64, 256, 3, 3, (1, 1), (1, 1)),      # one pair tile, halves partly past M
    synth.ConvShape(2, 28, 28, 128, 512, 3, 3, (1, 1), (1, 1)),     # 2 channel tiles, ragged M
    synth.ConvShape(1, 30, 30, 2048, 256, 1, 1, (1, 1), (0, 0)),    # plain GEMM, 32 K blocks
    synth.ConvShape(1, 16, 16, 64, 256, 7, 7, (1, 1), (3, 3)),      # 7x7 pad 3
    synth.ConvShape(2, 17, 17, 64, 256, 3, 3, (2, 2), (1, 1)),      # stride 2
    synth.ConvShape(1, 10, 30, 128, 256, 1, 1, (1, 1), (0, 0)),     # plain GEMM, short K: a half wholly past M
]


@pytest.mark.parametrize("variant", [4, 5], ids=["pair", "cta"])
@pytest.mark.parametrize("c", WIDE_SHAPES, ids=lambda c: f"{c.N}x{c.H}x{c.W}x{c.C_in}-{c.C_out}k{c.KH}s{c.stride[0]}")
def test_conv_umma_wide_small(b, c, variant):
    d = synth.conv_inputs(c, seed=16, w_dist="normal_fanin")
    got = _run_conv(b, c, d, variant)
    ref = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], c.stride, c.pad)
    _conv_check(got, ref)
    _assert_no_device_error(b)


def test_conv_umma_wide_two_waves_sampled(b):
    # 65536 pixels, 256 channels: 128 pair tiles over the GPU's pairs, a full
    # wave and a partial one too large to split into halves
    c = synth.ConvShape(16, 64, 64, 64, 256, 3, 3, (1, 1), (1, 1))
    d = synth.conv_inputs(c, seed=17, w_dist="normal_fanin")
    got = _run_conv(b, c, d, b.TF_CONV_UMMA_PAIR_WIDE).reshape(-1)
    pts = conv_sample_points(c.N, c.Ho, c.Wo, c.C_out, 4000, seed=5)
    ref = oracle.conv2d_bn_silu_points(d["x"], d["w_oihw"], d["scale"], d["bias"], pts, c.stride, c.pad)
    _conv_check(got[pts], ref)
    assert np.isfinite(got).all()
    _assert_no_device_error(b)


# One wave of wide tiles and a few more: the few (at most half a wave) run as
# a second launch on 128-row tiles, from the first row the wide launch leaves
# (ragged M: 11 x 61 x 61 = 40931 pixels).  Every output is checked.
WIDE_TAIL_SHAPES = [
    synth.ConvShape(11, 61, 61, 64, 256, 3, 3, (1, 1), (1, 1)),
    synth.ConvShape(11, 61, 61, 128, 256, 1, 1, (1, 1), (0, 0)),
]


@pytest.mark.parametrize("variant", [4, 5], ids=["pair", "cta"])
@pytest.mark.parametrize("c", WIDE_TAIL_SHAPES, ids=["3x3", "1x1"])
def test_conv_umma_wide_tail_launch(b, c, variant):
    d = synth.conv_inputs(c, seed=18, w_dist="normal_fanin")
    n0 = b.tf_launch_count()
    got = _run_conv(b, c, d, variant)
    conv_kernels = b.tf_launch_count() - n0 - 1   # less the filter pack
    # 80 pair tiles (160 single-CTA tiles): two launches on a GPU whose pairs
    # (CTAs) leave a partial wave of at most half, as GB300's do
    assert conv_kernels in (1, 2)
    if torch.cuda.get_device_properties(0).multi_processor_count >= 148:
        assert conv_kernels == 2
    ref = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], c.stride, c.pad)
    _conv_check(got, ref)
    _assert_no_device_error(b)


def test_conv_umma_wide_rejects_other_channel_counts(b):
    c = synth.ConvShape(1, 12, 12, 64, 128, 3, 3, (1, 1), (1, 1))
    x = torch.zeros((c.N, c.H, c.W, c.C_in), dtype=torch.int16, device="cuda")
    w = torch.zeros((c.C_out, c.KH, c.KW, c.C_in), dtype=torch.int16, device="cuda")
    sc = torch.ones((c.C_out,), dtype=torch.float32, device="cuda")
    y = torch.zeros((c.M, c.C_out), dtype=torch.int16, device="cuda")
    rc = b.tf_conv2d_bn_silu_variant(x, w, sc, sc, y, _shape(b, c), b.TF_CONV_UMMA_PAIR_WIDE, check=False)
    assert rc == b.TF_ERR_UNSUPPORTED


SPLITK_SHAPES = [
    synth.ConvShape(1, 16, 16, 256, 256, 3, 3, (1, 1), (1, 1)),     # 2 tiles, 36 K blocks
    synth.ConvShape(1, 8, 8, 512, 128, 3, 3, (1, 1), (1, 1)),       # one ragged tile
    synth.ConvShape(2, 14, 14, 128, 64, 7, 7, (1, 1), (3, 3)),      # 7x7, ragged M tail
    synth.ConvShape(1, 12, 12, 1024, 512, 1, 1, (1, 1), (0, 0)),    # 1x1, 2 N tiles, 16 K blocks
    synth.ConvShape(1, 10, 10, 200, 128, 3, 3, (1, 1), (1, 1)),     # C_in 200 = 3 x 64 + 8: 36 K blocks
]


@pytest.mark.parametrize("c", SPLITK_SHAPES, ids=lambda c: f"{c.N}x{c.H}x{c.W}x{c.C_in}-{c.C_out}k{c.KH}")
def test_conv_split_k_workspace(b, c):
    d = synth.conv_inputs(c, seed=15, w_dist="normal_fanin")
    shape = _shape(b, c)
    need = b.tf_conv2d_bn_silu_workspace_size(shape)
    assert need > 0, "shape expected to split"
    ws = torch.full((need // 4,), float("nan"), dtype=torch.float32, device="cuda")   # every partial must be written
    x = dev_u16(d["x"])
    w = torch.empty((c.C_out, c.KH, c.KW, c.C_in), dtype=torch.int16, device="cuda")
    b.tf_pack_filter_nhwc(dev_u16(d["w_oihw"]), w, c.C_out, c.C_in, c.KH, c.KW)
    ref = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], c.stride, c.pad)
    for nbytes in (need, need - 16, 0):   # split, then too small a workspace: the unsplit path
        y = torch.full((c.M, c.C_out), 0x7FC0, dtype=torch.int16, device="cuda")
        b.tf_conv2d_bn_silu_ws(x, w, dev_f32(d["scale"]), dev_f32(d["bias"]), y, shape, ws if nbytes else None, nbytes)
        torch.cuda.synchronize()
        _conv_check(bf16_to_f64(host_u16(y)).reshape(ref.shape), ref)
    _assert_no_device_error(b)


def test_conv_umma_plain_epilogue_is_the_bare_conv(b):
    c = synth.ConvShape(2, 12, 12, 64, 64, 3, 3, (1, 1), (1, 1))
    d = synth.conv_inputs(c, seed=3, w_dist="normal_fanin")
    got = _run_conv(b, c, d, b.TF_CONV_UMMA, fused=False)
    ref = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], c.stride, c.pad, oracle.EPI_NONE)
    _conv_check(got, ref)


def test_conv_dispatch_tiny_workload(b):
    w = synth.WORKLOADS["conv3x3_tiny_1x16x16x8_to16"]
    c = w.conv
    d = synth.workload_inputs(w)
    got = _run_conv(b, c, d, b.TF_CONV_AUTO)
    ref = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], c.stride, c.pad)
    _conv_check(got, ref)


# ---------------------------------------------------------------- conv, full workloads, sampled

@pytest.mark.parametrize("variant", [-1, 2, 3, 4], ids=["auto", "cta", "pair", "wide"])
@pytest.mark.parametrize("name,nrand", [("conv1x1_32x56x56x256_to256", 6000), ("conv7x7_16x64x64x512_to512", 1500)])
def test_conv_full_workload_sampled(b, name, nrand, variant):
    w = synth.WORKLOADS[name]
    c = w.conv
    d = synth.workload_inputs(w)
    got = _run_conv(b, c, d, variant).reshape(-1)
    pts = conv_sample_points(c.N, c.Ho, c.Wo, c.C_out, nrand, seed=4)
    ref = oracle.conv2d_bn_silu_points(d["x"], d["w_oihw"], d["scale"], d["bias"], pts, c.stride, c.pad)
    _conv_check(got[pts], ref)
    assert np.isfinite(got).all()
    _assert_no_device_error(b)


# ---------------------------------------------------------------- producer -> consumer convs

@pytest.mark.parametrize("standalone", [False, True])
def test_producer_consumer_pair(b, standalone):
    # a 1x1 producer, BN+SiLU, then a 7x7 consumer: the activation either in
    # the producer's epilogue or as separate BN and SiLU kernels
    p = synth.ConvShape(2, 12, 12, 128, 64, 1, 1, (1, 1), (0, 0))
    c = synth.ConvShape(2, 12, 12, 64, 64, 7, 7, (1, 1), (3, 3))
    d = synth.producer_consumer_inputs(p, c, seed=14)
    w1 = torch.empty((p.C_out, 1, 1, p.C_in), dtype=torch.int16, device="cuda")
    w2 = torch.empty((c.C_out, 7, 7, c.C_in), dtype=torch.int16, device="cuda")
    b.tf_pack_filter_nhwc(dev_u16(d["w1_oihw"]), w1, p.C_out, p.C_in, 1, 1)
    b.tf_pack_filter_nhwc(dev_u16(d["w2_oihw"]), w2, c.C_out, c.C_in, 7, 7)
    s1, b1, s2, b2 = (dev_f32(d[k]) for k in ("scale1", "bias1", "scale2", "bias2"))
    x = dev_u16(d["x"])
    u = torch.empty((p.M, p.C_out), dtype=torch.int16, device="cuda")
    y = torch.empty((c.M, c.C_out), dtype=torch.int16, device="cuda")
    if standalone:
        t1, t2 = torch.empty_like(u), torch.empty_like(u)
        b.tf_unfused_conv2d(x, w1, t1, _shape(b, p), b.TF_CONV_UMMA)
        b.tf_unfused_bn(t1, s1, b1, t2, p.M, p.C_out)
        b.tf_unfused_silu(t2, u, p.M * p.C_out)
    else:
        b.tf_conv2d_bn_silu_variant(x, w1, s1, b1, u, _shape(b, p), b.TF_CONV_UMMA)
    b.tf_conv2d_bn_silu_variant(u, w2, s2, b2, y, _shape(b, c), b.TF_CONV_UMMA)
    torch.cuda.synchronize()
    epi = oracle.EPI_CHAIN if standalone else oracle.EPI_FUSED
    u_ref = oracle.conv2d_bn_silu(d["x"], d["w1_oihw"], d["scale1"], d["bias1"], p.stride, p.pad, epi)
    u_bits = synth.f32_to_bf16_bits(u_ref.astype(np.float32))       # the stored intermediate
    y_ref = oracle.conv2d_bn_silu(u_bits, d["w2_oihw"], d["scale2"], d["bias2"], c.stride, c.pad)
    _conv_check(bf16_to_f64(host_u16(u)).reshape(u_ref.shape), u_ref)
    _conv_check(bf16_to_f64(host_u16(y)).reshape(y_ref.shape), y_ref)


# ---------------------------------------------------------------- bias + GELU

# rows of up to 16384 columns take the bulk-copy ring (chunks of whole rows,
# ragged last chunks at 37x200 and 129x1032); wider rows the grid-stride kernel
@pytest.mark.parametrize("rows,cols", [(1, 8), (3, 24), (37, 200), (129, 1032), (8192, 8192), (5, 16384),
                                       (3, 16392), (2, 40000)])
def test_bias_gelu(b, rows, cols):
    d = synth.bias_gelu_inputs(rows, cols, seed=5)
    y = torch.empty((rows, cols), dtype=torch.float16, device="cuda")
    b.tf_bias_gelu(dev_f16(d["x"]), dev_f16(d["bias"]), y, rows, cols)
    torch.cuda.synchronize()
    ref = oracle.bias_gelu(d["x"], d["bias"])
    ulp = f16_ulp_distance(y.cpu().numpy().view(np.uint16), ref)
    assert ulp.max() <= 2, f"max {ulp.max()} ulp"


def test_bias_gelu_every_fp16_input(b):
    # every finite fp16 value of s, bias zero: the fp16 subnormal outputs of
    # the deep negative tail, +-0, and the largest magnitudes (+-65504)
    xs = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
    xs = xs[np.isfinite(xs)]
    xs = xs[: (xs.size // 8) * 8].reshape(-1, 8)
    y = torch.empty(xs.shape, dtype=torch.float16, device="cuda")
    b.tf_bias_gelu(dev_f16(xs), dev_f16(np.zeros(8, np.float16)), y, xs.shape[0], 8)
    torch.cuda.synchronize()
    ref = oracle.bias_gelu(xs, np.zeros(8, np.float16))
    ulp = f16_ulp_distance(y.cpu().numpy().view(np.uint16), ref)
    assert ulp.max() <= 2, f"max {ulp.max()} ulp at s={xs.reshape(-1)[ulp.reshape(-1).argmax()]}"


# ---------------------------------------------------------------- bias + GELU + row sum

# Row-sum tolerance: each term carries the GELU evaluation error (~1e-5
# relative) and, on the split path, the fp16 rounding of y (<= 2^-12
# relative); fp32 accumulation over <= 16384 terms in a shallow tree adds
# ~30 * 2^-24 relative.  Bound: 1e-3 * sum_j |y_j| + 1e-3, four times the
# worst case.
def _rowsum_check(rs_gpu, y_ref):
    bound = 1e-3 * np.abs(y_ref).sum(axis=1) + 1e-3
    err = np.abs(rs_gpu.astype(np.float64) - y_ref.sum(axis=1))
    assert np.all(err <= bound), f"worst row error {err.max():.4g} (bound {bound[err.argmax()]:.4g})"


# Widths across the tile kernel's row-tile shapes, ragged row counts, one
# row, two rows, and fewer row tiles than SMs.
@pytest.mark.parametrize("rows,cols", [(1, 8), (3, 200), (37, 1032), (300, 16384), (8192, 8192),
                                       (1000, 256), (129, 768), (77, 2048), (5, 16384), (2, 256)])
def test_bias_gelu_rowsum_fused(b, rows, cols):
    d = synth.bias_gelu_inputs(rows, cols, seed=10)
    y = torch.empty((rows, cols), dtype=torch.float16, device="cuda")
    rs = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
    b.tf_bias_gelu_rowsum(dev_f16(d["x"]), dev_f16(d["bias"]), y, rs, rows, cols)
    torch.cuda.synchronize()
    ref_y, ref_rs = oracle.bias_gelu_rowsum(d["x"], d["bias"])
    assert f16_ulp_distance(y.cpu().numpy().view(np.uint16), ref_y).max() <= 2
    _rowsum_check(rs.cpu().numpy(), ref_y)
    _assert_no_device_error(b)


@pytest.mark.parametrize("rows,cols", [(3, 200), (8192, 8192)])
def test_bias_gelu_rowsum_split(b, rows, cols):
    d = synth.bias_gelu_inputs(rows, cols, seed=11)
    y = torch.empty((rows, cols), dtype=torch.float16, device="cuda")
    rs = torch.empty((rows,), dtype=torch.float32, device="cuda")
    b.tf_bias_gelu(dev_f16(d["x"]), dev_f16(d["bias"]), y, rows, cols)
    b.tf_unfused_rowsum(y, rs, rows, cols)
    torch.cuda.synchronize()
    ref_y, _ = oracle.bias_gelu_rowsum(d["x"], d["bias"])
    _rowsum_check(rs.cpu().numpy(), ref_y)


def test_bias_gelu_beyond_2_to_31_elements(b):
    # 262144 x 8200 = 2.15e9 values: 64-bit offsets, one 16400-byte row per
    # chunk of the bulk-copy ring.  The rows repeat a seeded 4096-row block on
    # the device.
    rows, cols, block = 262144, 8200, 4096
    d = synth.bias_gelu_inputs(block, cols, seed=16)
    x = dev_f16(d["x"]).repeat(rows // block, 1)
    y = torch.empty((rows, cols), dtype=torch.float16, device="cuda")
    b.tf_bias_gelu(x, dev_f16(d["bias"]), y, rows, cols)
    torch.cuda.synchronize()
    del x
    ref = oracle.bias_gelu(d["x"], d["bias"])
    for r in (0, 1, block - 1, 131071, 200003, rows - 1):
        ulp = f16_ulp_distance(y[r].cpu().numpy().view(np.uint16), ref[r % block])
        assert ulp.max() <= 2, (r, ulp.max())
    _assert_no_device_error(b)


# ---------------------------------------------------------------- residual + LayerNorm

@pytest.mark.parametrize("rows,hidden", [(1, 8), (5, 200), (33, 4096), (7, 16384), (16384, 4096)])
def test_residual_layernorm(b, rows, hidden):
    d = synth.layernorm_inputs(rows, hidden, seed=6)
    y = torch.empty((rows, hidden), dtype=torch.float16, device="cuda")
    b.tf_residual_layernorm(dev_f16(d["act"]), dev_f16(d["res"]), dev_f32(d["gamma"]), dev_f32(d["beta"]), y,
                            rows, hidden, 1e-5)
    torch.cuda.synchronize()
    ref = oracle.residual_layernorm(d["act"], d["res"], d["gamma"], d["beta"], eps=1e-5)
    err = np.abs(y.cpu().numpy().astype(np.float64) - ref)
    assert err.max() <= 1e-2, err.max()


@pytest.mark.parametrize("variant,rows,hidden", [
    (0, 5, 8), (0, 37, 200), (0, 64, 1024), (0, 3, 1000),
    (1, 5, 8), (1, 9, 8200), (1, 4, 16384),
    (2, 3, 16392), (2, 5, 40000), (2, 2, 131072),
])
def test_layernorm_each_strategy(b, variant, rows, hidden):
    d = synth.layernorm_inputs(rows, hidden, seed=12)
    y = torch.empty((rows, hidden), dtype=torch.float16, device="cuda")
    b.tf_residual_layernorm_variant(dev_f16(d["act"]), dev_f16(d["res"]), dev_f32(d["gamma"]), dev_f32(d["beta"]),
                                    y, rows, hidden, 1e-5, variant)
    torch.cuda.synchronize()
    ref = oracle.residual_layernorm(d["act"], d["res"], d["gamma"], d["beta"], eps=1e-5)
    err = np.abs(y.cpu().numpy().astype(np.float64) - ref)
    assert err.max() <= 1e-2, err.max()
    _assert_no_device_error(b)


def test_layernorm_wide_rows_dispatch(b):
    rows, hidden = 6, 65536
    assert b.tf_residual_layernorm_select(hidden) == b.TF_LN_CLUSTER
    d = synth.layernorm_inputs(rows, hidden, seed=13)
    y = torch.empty((rows, hidden), dtype=torch.float16, device="cuda")
    b.tf_residual_layernorm(dev_f16(d["act"]), dev_f16(d["res"]), dev_f32(d["gamma"]), dev_f32(d["beta"]), y,
                            rows, hidden, 1e-5)
    torch.cuda.synchronize()
    ref = oracle.residual_layernorm(d["act"], d["res"], d["gamma"], d["beta"], eps=1e-5)
    assert np.abs(y.cpu().numpy().astype(np.float64) - ref).max() <= 1e-2


def test_layernorm_beyond_2_to_31_elements(b):
    # 262144 x 8200 = 2.15e9 values per tensor, rows repeating a seeded block
    rows, hidden, block = 262144, 8200, 2048
    d = synth.layernorm_inputs(block, hidden, seed=17)
    act = dev_f16(d["act"]).repeat(rows // block, 1)
    res = dev_f16(d["res"]).repeat(rows // block, 1)
    y = torch.empty((rows, hidden), dtype=torch.float16, device="cuda")
    b.tf_residual_layernorm(act, res, dev_f32(d["gamma"]), dev_f32(d["beta"]), y, rows, hidden, 1e-5)
    torch.cuda.synchronize()
    del act, res
    ref = oracle.residual_layernorm(d["act"], d["res"], d["gamma"], d["beta"], eps=1e-5)
    for r in (0, block - 1, 131071, 200003, rows - 1):
        assert np.abs(y[r].cpu().numpy().astype(np.float64) - ref[r % block]).max() <= 1e-2, r
    _assert_no_device_error(b)


def test_layernorm_constant_row(b):
    # variance 0: the output is beta exactly (0 * rsqrt(eps) * gamma + beta)
    rows, hidden = 4, 64
    act = np.full((rows, hidden), 1.5, np.float16)
    res = np.full((rows, hidden), -0.25, np.float16)
    gamma = np.linspace(0.5, 1.5, hidden).astype(np.float32)
    beta = np.linspace(-1, 1, hidden).astype(np.float32)
    y = torch.empty((rows, hidden), dtype=torch.float16, device="cuda")
    b.tf_residual_layernorm(dev_f16(act), dev_f16(res), dev_f32(gamma), dev_f32(beta), y, rows, hidden, 1e-5)
    torch.cuda.synchronize()
    ref = oracle.residual_layernorm(act, res, gamma, beta, eps=1e-5)
    assert np.abs(y.cpu().numpy().astype(np.float64) - ref).max() <= 1e-2


# ---------------------------------------------------------------- unfused chains

def test_unfused_conv_chain(b):
    c = synth.ConvShape(2, 12, 12, 64, 64, 3, 3, (1, 1), (1, 1))
    d = synth.conv_inputs(c, seed=7, w_dist="normal_fanin")
    x = dev_u16(d["x"])
    w = torch.empty((c.C_out, c.KH, c.KW, c.C_in), dtype=torch.int16, device="cuda")
    b.tf_pack_filter_nhwc(dev_u16(d["w_oihw"]), w, c.C_out, c.C_in, c.KH, c.KW)
    M = c.N * c.Ho * c.Wo
    t1 = torch.empty((M, c.C_out), dtype=torch.int16, device="cuda")
    t2 = torch.empty_like(t1)
    y = torch.empty_like(t1)
    b.tf_unfused_conv2d(x, w, t1, _shape(b, c), b.TF_CONV_UMMA)
    b.tf_unfused_bn(t1, dev_f32(d["scale"]), dev_f32(d["bias"]), t2, M, c.C_out)
    b.tf_unfused_silu(t2, y, M * c.C_out)
    torch.cuda.synchronize()
    ref = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], c.stride, c.pad, oracle.EPI_CHAIN)
    _conv_check(bf16_to_f64(host_u16(y)).reshape(ref.shape), ref)


def test_unfused_gelu_chain(b):
    rows, cols = 64, 1024
    d = synth.bias_gelu_inputs(rows, cols, seed=8)
    t = torch.empty((rows, cols), dtype=torch.float16, device="cuda")
    y = torch.empty_like(t)
    b.tf_unfused_bias_add(dev_f16(d["x"]), dev_f16(d["bias"]), t, rows, cols)
    b.tf_unfused_gelu(t, y, rows * cols)
    torch.cuda.synchronize()
    ref = oracle.bias_gelu(d["x"], d["bias"], materialize=True)
    ulp = f16_ulp_distance(y.cpu().numpy().view(np.uint16), ref)
    assert ulp.max() <= 2


def test_unfused_layernorm_chain(b):
    rows, hidden = 64, 4096
    d = synth.layernorm_inputs(rows, hidden, seed=9)
    s = torch.empty((rows, hidden), dtype=torch.float16, device="cuda")
    n = torch.empty_like(s)
    y = torch.empty_like(s)
    b.tf_unfused_residual_add(dev_f16(d["act"]), dev_f16(d["res"]), s, rows * hidden)
    b.tf_unfused_layernorm(s, n, rows, hidden, 1e-5)
    b.tf_unfused_affine(n, dev_f32(d["gamma"]), dev_f32(d["beta"]), y, rows, hidden)
    torch.cuda.synchronize()
    ref = oracle.residual_layernorm(d["act"], d["res"], d["gamma"], d["beta"], eps=1e-5, materialize=True)
    assert np.abs(y.cpu().numpy().astype(np.float64) - ref).max() <= 1e-2


# ---------------------------------------------------------------- stream order under programmatic launch
#
# Every kernel is launched with programmatic dependent launch and waits
# (griddepcontrol.wait) before its first global-memory access.  These calls
# run back to back on one stream without a host synchronisation between
# them; a kernel that started touching memory too early would read a
# half-written input (read after write) or overwrite an input the previous
# kernel is still reading (write after read).

def test_stream_order_read_after_write(b):
    rows, cols = 4096, 8192
    d0 = synth.bias_gelu_inputs(rows, cols, seed=30)
    d1 = synth.bias_gelu_inputs(rows, cols, seed=31)
    x = dev_f16(d0["x"])
    y1 = torch.full((rows, cols), float("nan"), dtype=torch.float16, device="cuda")
    y2 = torch.empty_like(y1)
    y3 = torch.empty_like(y1)
    g, be = dev_f32(np.ones(cols, np.float32)), dev_f32(d1["bias"].astype(np.float32))
    for _ in range(3):
        b.tf_bias_gelu(x, dev_f16(d0["bias"]), y1, rows, cols)      # y1 = GELU(x + b0)
        b.tf_bias_gelu(y1, dev_f16(d1["bias"]), y2, rows, cols)     # reads y1 at once
        b.tf_residual_layernorm(y2, y1, g, be, y3, rows, cols, 1e-5)   # reads both
    torch.cuda.synchronize()
    h1 = y1.cpu().numpy()
    h2 = y2.cpu().numpy()
    assert f16_ulp_distance(h2.view(np.uint16), oracle.bias_gelu(h1, d1["bias"])).max() <= 2
    ref3 = oracle.residual_layernorm(h2, h1, np.ones(cols, np.float32), d1["bias"].astype(np.float32), eps=1e-5)
    assert np.abs(y3.cpu().numpy().astype(np.float64) - ref3).max() <= 1e-2
    _assert_no_device_error(b)


def test_stream_order_write_after_read(b):
    rows, cols = 4096, 8192
    d0 = synth.bias_gelu_inputs(rows, cols, seed=32)
    d1 = synth.bias_gelu_inputs(rows, cols, seed=33)
    x = dev_f16(d0["x"])
    z = dev_f16(d1["x"])
    bias = dev_f16(d0["bias"])
    y = torch.empty((rows, cols), dtype=torch.float16, device="cuda")
    b.tf_bias_gelu(x, bias, y, rows, cols)   # reads x ...
    b.tf_bias_gelu(z, bias, x, rows, cols)   # ... which the next call overwrites
    torch.cuda.synchronize()
    assert f16_ulp_distance(y.cpu().numpy().view(np.uint16), oracle.bias_gelu(d0["x"], d0["bias"])).max() <= 2
    assert f16_ulp_distance(x.cpu().numpy().view(np.uint16), oracle.bias_gelu(d1["x"], d0["bias"])).max() <= 2


def test_stream_order_conv_chain(b):
    # the tensor-core conv's output feeds the next conv, whose output then
    # overwrites the first conv's input
    c = synth.ConvShape(2, 28, 28, 128, 128, 1, 1, (1, 1), (0, 0))
    d = synth.conv_inputs(c, seed=34, w_dist="normal_fanin")
    x = dev_u16(d["x"])
    w = torch.empty((c.C_out, 1, 1, c.C_in), dtype=torch.int16, device="cuda")
    b.tf_pack_filter_nhwc(dev_u16(d["w_oihw"]), w, c.C_out, c.C_in, 1, 1)
    sc, bi = dev_f32(d["scale"]), dev_f32(d["bias"])
    shape = _shape(b, c)
    y1 = torch.empty((c.M, c.C_out), dtype=torch.int16, device="cuda")
    b.tf_conv2d_bn_silu_variant(x, w, sc, bi, y1, shape, b.TF_CONV_UMMA)
    b.tf_conv2d_bn_silu_variant(y1, w, sc, bi, x, shape, b.TF_CONV_UMMA)   # reads y1, overwrites x
    torch.cuda.synchronize()
    h1 = host_u16(y1).reshape(c.N, c.Ho, c.Wo, c.C_out)   # bf16 words
    ref1 = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], c.stride, c.pad)
    _conv_check(bf16_to_f64(h1), ref1)
    ref2 = oracle.conv2d_bn_silu(h1, d["w_oihw"], d["scale"], d["bias"], c.stride, c.pad)
    _conv_check(bf16_to_f64(host_u16(x)).reshape(ref2.shape), ref2)
    _assert_no_device_error(b)


# ---------------------------------------------------------------- bounded waits

def test_wait_probe_times_out_and_context_survives(b):
    _assert_no_device_error(b)
    b.tf_wait_probe(2_000_000)   # 2 ms on a barrier nothing arrives on
    rc, word = b.tf_read_device_error()
    assert rc == b.TF_ERR_TIMEOUT and word == b.TF_DEVERR_PROBE_WAIT
    _assert_no_device_error(b)   # the word was cleared
    test_conv_umma_plain_epilogue_is_the_bare_conv(b)   # the context still works
