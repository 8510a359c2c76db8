"""The C-ABI library builds, loads and exports every declared entry point, and
rejects bad arguments on the host before launching anything (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tf_epilogue.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(tf_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("tf_pack_filter_nhwc", "tf_conv2d_bn_silu", "tf_bias_gelu", "tf_residual_layernorm"):
        assert required in names


def test_library_exports_every_declared_symbol(native_lib):
    from gemm_conv_epilogues_gb300 import binding
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (tf_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(native_lib, n)


def test_launch_counter_counts_nothing_rejected_on_the_host(native_lib):
    from gemm_conv_epilogues_gb300 import binding as b
    n0 = b.tf_launch_count()
    assert b.tf_bias_gelu(0, 0, 0, 8, 8, 0, check=False) == b.TF_ERR_INVALID_ARG
    assert b.tf_launch_count() == n0


def test_status_strings(native_lib):
    from gemm_conv_epilogues_gb300 import binding as b
    assert b.status_string(0) == "TF_OK"
    for s in (1, 2, 3, 4):
        assert b.status_string(s).startswith("TF_ERR_")


def test_wait_limit_round_trip(native_lib):
    from gemm_conv_epilogues_gb300 import binding as b
    old = b.tf_get_wait_limit_ns()
    try:
        b.tf_set_wait_limit_ns(12345)
        assert b.tf_get_wait_limit_ns() == 12345
    finally:
        b.tf_set_wait_limit_ns(old)


def test_host_validation_rejects_before_launch(native_lib):
    from gemm_conv_epilogues_gb300 import binding as b
    S = b.TF_ERR_INVALID_ARG
    U = b.TF_ERR_UNSUPPORTED
    p16 = 1 << 20           # a 16-byte aligned fake address; never dereferenced on these paths
    odd = p16 + 2
    shape = b.conv_shape(1, 16, 16, 8, 16, 3, 3, (1, 1), (1, 1))
    assert b.tf_conv2d_bn_silu(None, p16, p16, p16, p16, shape, 0, check=False) == S
    assert b.tf_conv2d_bn_silu(p16, p16, None, p16, p16, shape, 0, check=False) == S
    assert b.tf_conv2d_bn_silu(odd, p16, p16, p16, p16, shape, 0, check=False) == U
    bad = b.conv_shape(1, 16, 16, 12, 16, 3, 3, (1, 1), (1, 1))          # C_in % 8 != 0
    assert b.tf_conv2d_bn_silu(p16, p16, p16, p16, p16, bad, 0, check=False) == U
    empty = b.conv_shape(1, 2, 2, 8, 16, 5, 5, (1, 1), (0, 0))           # no output pixel
    assert b.tf_conv2d_bn_silu(p16, p16, p16, p16, p16, empty, 0, check=False) == S
    zero = b.conv_shape(0, 16, 16, 8, 16, 3, 3, (1, 1), (1, 1))
    assert b.tf_conv2d_bn_silu(p16, p16, p16, p16, p16, zero, 0, check=False) == S
    assert b.tf_conv2d_bn_silu_variant(p16, p16, p16, p16, p16, shape, 7, 0, check=False) == S
    # the paired tensor-core kernel needs whole 32-channel tiles (C_out 16 here);
    # rejected on the host before any launch
    assert b.tf_conv2d_bn_silu_variant(p16, p16, p16, p16, p16, shape, b.TF_CONV_UMMA_PAIR, 0, check=False) == U
    assert b.tf_bias_gelu(p16, p16, p16, 0, 8, 0, check=False) == S
    assert b.tf_bias_gelu(p16, None, p16, 4, 8, 0, check=False) == S
    assert b.tf_bias_gelu(p16, p16, p16, 4, 12, 0, check=False) == U
    assert b.tf_bias_gelu(p16, p16, odd, 4, 8, 0, check=False) == U
    assert b.tf_residual_layernorm(p16, p16, p16, p16, p16, 4, 0, 1e-5, 0, check=False) == S
    assert b.tf_residual_layernorm(p16, p16, p16, p16, p16, 4, 8, -1.0, 0, check=False) == S
    assert b.tf_residual_layernorm(p16, p16, p16, p16, p16, 4, 20, 1e-5, 0, check=False) == U
    assert b.tf_residual_layernorm(p16, p16, p16, p16, p16, 4, 262144, 1e-5, 0, check=False) == U
    assert b.tf_residual_layernorm_variant(p16, p16, p16, p16, p16, 4, 64, 1e-5, 5, 0, check=False) == S
    assert b.tf_residual_layernorm_select(512) == b.TF_LN_WARP
    assert b.tf_residual_layernorm_select(4096) == b.TF_LN_CTA
    assert b.tf_residual_layernorm_select(65536) == b.TF_LN_CLUSTER
    assert b.tf_residual_layernorm_select(262144) == -b.TF_ERR_UNSUPPORTED
    assert b.tf_residual_layernorm_select(100) == -b.TF_ERR_UNSUPPORTED
    assert b.tf_bias_gelu_rowsum(p16, p16, p16, None, 4, 8, 0, check=False) == S
    assert b.tf_bias_gelu_rowsum(p16, p16, p16, p16, 4, 32768, 0, check=False) == U
    assert b.tf_unfused_rowsum(p16, p16, 4, 12, 0, check=False) == U
    assert b.tf_pack_filter_nhwc(None, p16, 4, 4, 3, 3, 0, check=False) == S
    assert b.tf_pack_filter_nhwc(p16, p16, 0, 4, 3, 3, 0, check=False) == S
    assert b.tf_unfused_bn(p16, p16, p16, p16, 4, 12, 0, check=False) == U
    assert b.tf_unfused_silu(p16, p16, 0, 0, check=False) == S
    assert b.tf_unfused_gelu(p16, odd, 8, 0, check=False) == U
    assert b.tf_unfused_residual_add(p16, p16, p16, 12, 0, check=False) == U
    assert b.tf_unfused_layernorm(p16, p16, 2, 10, 1e-5, 0, check=False) == U
    assert b.tf_unfused_affine(p16, p16, p16, None, 2, 8, 0, check=False) == S
    # per-channel parameters read as 16-byte vectors must be aligned
    quad = p16 + 4   # 4-byte aligned, as a float array can be
    assert b.tf_unfused_bn(p16, quad, p16, p16, 4, 8, 0, check=False) == U
    assert b.tf_unfused_bn(p16, p16, quad, p16, 4, 8, 0, check=False) == U
    assert b.tf_unfused_affine(p16, quad, p16, p16, 2, 8, 0, check=False) == U
    assert b.tf_unfused_affine(p16, p16, quad, p16, 2, 8, 0, check=False) == U
    assert b.tf_unfused_bias_add(p16, odd, p16, 2, 8, 0, check=False) == U
    assert b.tf_residual_layernorm(p16, p16, quad, p16, p16, 4, 64, 1e-5, 0, check=False) == U


def test_split_k_workspace_size(native_lib):
    from gemm_conv_epilogues_gb300 import binding as b, synth
    big = synth.WORKLOADS["conv7x7_16x64x64x512_to512"].conv
    assert b.tf_conv2d_bn_silu_workspace_size(b.conv_shape(big.N, big.H, big.W, big.C_in, big.C_out, 7, 7,
                                                           (1, 1), (3, 3))) == 0
    small = b.conv_shape(1, 16, 16, 256, 256, 3, 3, (1, 1), (1, 1))      # 2 output tiles, 36 K blocks
    need = b.tf_conv2d_bn_silu_workspace_size(small)
    assert need > 0 and need % (256 * 256 * 4) == 0
    assert b.tf_conv2d_bn_silu_workspace_size(b.conv_shape(1, 16, 16, 8, 16, 3, 3, (1, 1), (1, 1))) == 0
    p16 = 1 << 20
    assert b.tf_conv2d_bn_silu_ws(p16, p16, p16, p16, p16, small, None, 64, 0, check=False) == b.TF_ERR_INVALID_ARG
    assert b.tf_conv2d_bn_silu_ws(p16, p16, p16, p16, p16, small, p16 + 8, need, 0, check=False) == \
        b.TF_ERR_UNSUPPORTED


def test_dispatch_selects_by_shape(native_lib):
    from gemm_conv_epilogues_gb300 import binding as b, synth
    w = synth.WORKLOADS
    sel = lambda c: b.tf_conv2d_bn_silu_select(b.conv_shape(c.N, c.H, c.W, c.C_in, c.C_out, c.KH, c.KW, c.stride, c.pad))
    assert sel(w["conv3x3_tiny_1x16x16x8_to16"].conv) == b.TF_CONV_DIRECT
    assert sel(w["conv1x1_32x56x56x256_to256"].conv) == b.TF_CONV_UMMA
    assert sel(w["conv7x7_16x64x64x512_to512"].conv) == b.TF_CONV_UMMA_PAIR_WIDE   # long K, many 256-channel tiles
    assert sel(synth.ConvShape(16, 64, 64, 512, 128, 7, 7, (1, 1), (3, 3))) == b.TF_CONV_UMMA   # 128 channels
    assert sel(synth.ConvShape(1, 64, 64, 512, 256, 7, 7, (1, 1), (3, 3))) == b.TF_CONV_UMMA   # too few tiles
    # short K with 256 channels over two waves: paired MMA (single CTAs would take 128-channel tiles)
    assert sel(synth.ConvShape(16, 64, 64, 64, 256, 3, 3, (1, 1), (1, 1))) == b.TF_CONV_UMMA_PAIR
    assert sel(synth.ConvShape(16, 64, 64, 256, 256, 1, 1)) == b.TF_CONV_UMMA   # plain 1x1: resident filters
    assert sel(synth.ConvShape(1, 16, 16, 64, 256, 1, 1)) == b.TF_CONV_UMMA   # 8.4 MFLOP: tensor cores win
    # channel tails run on the tensor cores too (C_in >= 16 or enough work)
    assert sel(synth.ConvShape(16, 32, 32, 24, 48, 3, 3, (1, 1), (1, 1))) == b.TF_CONV_UMMA
    assert sel(synth.ConvShape(4, 32, 32, 256, 16, 3, 3, (1, 1), (1, 1))) == b.TF_CONV_UMMA
    assert sel(synth.ConvShape(16, 64, 64, 24, 128, 3, 3, (1, 1), (1, 1))) == b.TF_CONV_UMMA_PAIR   # C_in tail
    assert sel(synth.ConvShape(4, 32, 32, 8, 64, 3, 3, (1, 1), (1, 1))) == b.TF_CONV_UMMA
    # few input channels and few outputs stay on the CUDA cores
    assert sel(synth.ConvShape(4, 32, 32, 8, 32, 3, 3, (1, 1), (1, 1))) == b.TF_CONV_DIRECT
    assert sel(synth.ConvShape(16, 64, 64, 8, 32, 3, 3, (1, 1), (1, 1))) == b.TF_CONV_TILED
    # small 3x3 layers over few input channels: the direct kernel's batched tap loads
    assert sel(synth.ConvShape(1, 16, 16, 24, 128, 3, 3, (1, 1), (1, 1))) == b.TF_CONV_DIRECT
    assert sel(synth.ConvShape(4, 32, 32, 24, 16, 3, 3, (1, 1), (1, 1))) == b.TF_CONV_UMMA   # 64K outputs
    # tiny reductions stay on the direct kernel even when the tensor-core one could run
    assert sel(synth.ConvShape(1, 16, 16, 64, 64, 1, 1)) == b.TF_CONV_DIRECT
    assert sel(synth.ConvShape(1, 16, 16, 256, 64, 1, 1)) == b.TF_CONV_UMMA
    assert b.tf_conv2d_bn_silu_select(b.conv_shape(1, 2, 2, 8, 16, 5, 5)) == -b.TF_ERR_INVALID_ARG
