"""GPU parity on the two full-size convolution workloads, EVERY output
element against the fp64 oracle, in the launch configuration the bench times
(tf_conv2d_bn_silu, kernel chosen by the shape dispatch).

"Fusing an Epilogue", "When not to fuse": the fused kernel has to be checked
against what it replaces on the shapes that actually run, so these compare
the whole output tensor, not a sample.  The oracle needs about 0.3 s (1x1,
13.2 GFLOP) and 40-60 s (7x7, 1.68 TFLOP in fp64) on 16 host cores.

Tolerance (bf16 output): |gpu - ref| <= 1e-2 + 1e-2*|ref|.
"""
import numpy as np
import pytest
import torch

import oracle
from gemm_conv_epilogues_gb300 import synth
from helpers import bf16_to_f64, dev_f32, dev_u16, host_u16

pytestmark = pytest.mark.gpu

CONV_ATOL, CONV_RTOL = 1e-2, 1e-2


@pytest.fixture(scope="module")
def b(cuda_ready):
    from gemm_conv_epilogues_gb300 import binding
    return binding


@pytest.mark.parametrize("name", ["conv1x1_32x56x56x256_to256", "conv7x7_16x64x64x512_to512"])
def test_conv_full_workload_every_output(b, name):
    w = synth.WORKLOADS[name]
    c = w.conv
    d = synth.workload_inputs(w)
    x = dev_u16(d["x"])
    wt = torch.empty((c.C_out, c.KH, c.KW, c.C_in), dtype=torch.int16, device="cuda")
    b.tf_pack_filter_nhwc(dev_u16(d["w_oihw"]), wt, c.C_out, c.C_in, c.KH, c.KW)
    y = torch.full((c.N, c.Ho, c.Wo, c.C_out), 0x7FC0, dtype=torch.int16, device="cuda")   # NaN sentinel
    shape = b.conv_shape(c.N, c.H, c.W, c.C_in, c.C_out, c.KH, c.KW, c.stride, c.pad)
    b.tf_conv2d_bn_silu(x, wt, dev_f32(d["scale"]), dev_f32(d["bias"]), y, shape)
    torch.cuda.synchronize()
    rc, word = b.tf_read_device_error()
    assert rc == b.TF_OK and word == 0, (rc, hex(word))
    got = bf16_to_f64(host_u16(y))
    ref = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], c.stride, c.pad)
    assert got.shape == ref.shape
    err = np.abs(got - ref)
    bad = ~(err <= CONV_ATOL + CONV_RTOL * np.abs(ref))   # NaN (an unwritten output) counts as bad
    assert not bad.any(), (f"{int(bad.sum())} of {bad.size} outputs outside tolerance; "
                           f"first at flat index {int(np.flatnonzero(bad)[0])}; worst {np.nanmax(err):.4g}")
