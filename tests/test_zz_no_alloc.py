"""tf_conv2d_bn_silu_static_ws: the split-K conv for callers that cannot
allocate device memory -- a serving runtime or plugin host that owns every
device buffer, or code that must not call cudaMalloc while it serves.

Checked through the C ABI against the fp64 oracle (same tolerance as every
conv test: |gpu - ref| <= 1e-2 + 1e-2*|ref|) on consecutive calls that reuse
the library's static partial-sum array, on a fresh stream, and for its
contract that a call allocates no device memory.  Collected last on purpose,
so that a run stopping at the first failure has already run every other
test; it passes alone in a fresh process as well."""
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


def _setup(b, c, seed):
    d = synth.conv_inputs(c, seed=seed, w_dist="normal_fanin")
    w = torch.empty((c.C_out, c.KH, c.KW, c.C_in), dtype=torch.int16, device="cuda")
    b.tf_pack_filter_nhwc(dev_u16(d["w_oihw"]), w, c.C_out, c.C_in, c.KH, c.KW)
    shape = b.conv_shape(c.N, c.H, c.W, c.C_in, c.C_out, c.KH, c.KW, c.stride, c.pad)
    ref = oracle.conv2d_bn_silu(d["x"], d["w_oihw"], d["scale"], d["bias"], c.stride, c.pad)
    return dev_u16(d["x"]), w, dev_f32(d["scale"]), dev_f32(d["bias"]), shape, ref.reshape(c.M, c.C_out)


def _check(y, ref):
    got = bf16_to_f64(host_u16(y))
    assert np.all(np.abs(got - ref) <= CONV_ATOL + CONV_RTOL * np.abs(ref))   # NaN fails too


# two different split shapes: 2 tiles x 36 K blocks, and a 7x7 with a ragged M tail
CASES = [synth.ConvShape(1, 16, 16, 256, 256, 3, 3, (1, 1), (1, 1)),
         synth.ConvShape(2, 14, 14, 128, 64, 7, 7, (1, 1), (3, 3))]


def test_static_workspace_matches_oracle_on_consecutive_calls(b):
    # the shapes alternate, so every call after the first reuses an array
    # that another shape's partial sums filled
    for i, c in enumerate(CASES * 2):
        x, w, sc, bi, shape, ref = _setup(b, c, seed=20 + i)
        need = b.tf_conv2d_bn_silu_workspace_size(shape)
        assert 0 < need <= 8 << 20, "shape expected to split within the static array"
        for _ in range(2):   # two calls in a row on the same shape
            y = torch.full((c.M, c.C_out), 0x7FC0, dtype=torch.int16, device="cuda")   # NaN sentinel
            b.tf_conv2d_bn_silu_static_ws(x, w, sc, bi, y, shape)
            torch.cuda.synchronize()
            _check(y, ref)
    rc, word = b.tf_read_device_error()
    assert rc == b.TF_OK and word == 0


def test_static_workspace_allocates_nothing_and_runs_on_a_fresh_stream(b):
    c = CASES[0]
    x, w, sc, bi, shape, ref = _setup(b, c, seed=25)
    y = torch.full((c.M, c.C_out), 0x7FC0, dtype=torch.int16, device="cuda")
    y2 = torch.full((c.M, c.C_out), 0x7FC0, dtype=torch.int16, device="cuda")
    stream = torch.cuda.Stream()
    # the first call in a process looks the array's address up (and may load
    # the library's module); measure from after it
    b.tf_conv2d_bn_silu_static_ws(x, w, sc, bi, y, shape)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        b.tf_conv2d_bn_silu_static_ws(x, w, sc, bi, y, shape)
    # a stream the library has not seen before: the cached address serves it
    b.tf_conv2d_bn_silu_static_ws(x, w, sc, bi, y2, shape, stream=stream)
    stream.synchronize()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes across the calls"
    _check(y, ref)
    _check(y2, ref)
    rc, word = b.tf_read_device_error()
    assert rc == b.TF_OK and word == 0


def test_static_workspace_rejects_oversized_split(b):
    # 1024 pixels x 1024 channels with 36 K blocks splits 4 ways: 16 MiB of
    # partial sums, more than the 8 MiB array
    c = synth.ConvShape(1, 32, 32, 256, 1024, 3, 3, (1, 1), (1, 1))
    d = synth.conv_inputs(c, seed=30, w_dist="normal_fanin")
    w = torch.empty((c.C_out, c.KH, c.KW, c.C_in), dtype=torch.int16, device="cuda")
    b.tf_pack_filter_nhwc(dev_u16(d["w_oihw"]), w, c.C_out, c.C_in, c.KH, c.KW)
    shape = b.conv_shape(c.N, c.H, c.W, c.C_in, c.C_out, c.KH, c.KW, c.stride, c.pad)
    need = b.tf_conv2d_bn_silu_workspace_size(shape)
    assert need > 8 << 20
    y = torch.empty((c.M, c.C_out), dtype=torch.int16, device="cuda")
    rc = b.tf_conv2d_bn_silu_static_ws(dev_u16(d["x"]), w, dev_f32(d["scale"]), dev_f32(d["bias"]), y, shape,
                                       check=False)
    assert rc == b.TF_ERR_UNSUPPORTED
