"""tf_conv2d_bn_silu_static_ws: the split-K conv for callers that cannot
allocate device memory (a runtime that owns every buffer, or code that must
not call cudaMalloc while serving), checked through the C ABI against the
workspace-taking entry point tf_conv2d_bn_silu_ws, on two calls in a row.
Collected last on purpose so that a run stopping at the first failure has
already run every other test."""
import numpy as np
import pytest
import torch

from gemm_conv_epilogues_gb300 import synth
from helpers import bf16_to_f64, dev_f32, dev_u16, host_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def b(cuda_ready):
    from gemm_conv_epilogues_gb300 import binding
    return binding


def _setup(b, c, seed):
    d = synth.conv_inputs(c, seed=seed, w_dist="normal_fanin")
    w = torch.empty((c.C_out, c.KH, c.KW, c.C_in), dtype=torch.int16, device="cuda")
    b.tf_pack_filter_nhwc(dev_u16(d["w_oihw"]), w, c.C_out, c.C_in, c.KH, c.KW)
    shape = b.conv_shape(c.N, c.H, c.W, c.C_in, c.C_out, c.KH, c.KW, c.stride, c.pad)
    return dev_u16(d["x"]), w, dev_f32(d["scale"]), dev_f32(d["bias"]), shape


def test_static_workspace_matches_caller_workspace_on_consecutive_calls(b):
    # two different split shapes back to back: the second call reuses the
    # array the first one filled
    cases = [synth.ConvShape(1, 16, 16, 256, 256, 3, 3, (1, 1), (1, 1)),
             synth.ConvShape(2, 14, 14, 128, 64, 7, 7, (1, 1), (3, 3))]
    for i, c in enumerate(cases * 2):
        x, w, sc, bi, shape = _setup(b, c, seed=20 + i)
        need = b.tf_conv2d_bn_silu_workspace_size(shape)
        assert 0 < need <= 8 << 20
        ws = torch.empty((need // 4,), dtype=torch.float32, device="cuda")
        y_ref = torch.empty((c.M, c.C_out), dtype=torch.int16, device="cuda")
        y = torch.full((c.M, c.C_out), 0x7FC0, dtype=torch.int16, device="cuda")
        b.tf_conv2d_bn_silu_ws(x, w, sc, bi, y_ref, shape, ws, need)
        b.tf_conv2d_bn_silu_static_ws(x, w, sc, bi, y, shape)
        torch.cuda.synchronize()
        got, ref = bf16_to_f64(host_u16(y)), bf16_to_f64(host_u16(y_ref))
        assert np.all(np.abs(got - ref) <= 1e-2 + 1e-2 * np.abs(ref))
    rc, word = b.tf_read_device_error()
    assert rc == b.TF_OK and word == 0


def test_static_workspace_rejects_oversized_split(b):
    # 1024 pixels x 1024 channels with 36 K blocks splits 4 ways: 16 MiB of
    # partial sums, more than the 8 MiB array
    c = synth.ConvShape(1, 32, 32, 256, 1024, 3, 3, (1, 1), (1, 1))
    x, w, sc, bi, shape = _setup(b, c, seed=30)
    need = b.tf_conv2d_bn_silu_workspace_size(shape)
    assert need > 8 << 20
    y = torch.empty((c.M, c.C_out), dtype=torch.int16, device="cuda")
    assert b.tf_conv2d_bn_silu_static_ws(x, w, sc, bi, y, shape, check=False) == b.TF_ERR_UNSUPPORTED
