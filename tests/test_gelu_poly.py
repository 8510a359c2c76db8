"""The GELU kernels' polynomial, pinned on the CPU: the coefficients committed
in csrc/gelu_poly.h, evaluated step by step as the kernels do in fp32
(clamp, Horner in t, 2^P, max(s - s*Q, s*Q)), against s*Phi(s) from scipy on
every finite fp16 input -- within 1 fp16 ulp of the correctly rounded value
(the GPU tests allow 2)."""
import os
import re
import sys

import numpy as np
import pytest

CSRC = os.path.join(os.path.dirname(__file__), "..", "gemm_conv_epilogues_gb300", "csrc")


def _header_coefficients():
    text = open(os.path.join(CSRC, "gelu_poly.h")).read()
    deg = int(re.search(r"#define TF_GELU_POLY_DEGREE (\d+)", text).group(1))
    coef = [float(re.search(rf"#define TF_GELU_C{k} (\S+)f\n", text).group(1)) for k in range(deg + 1)]
    clamp = float(re.search(r"#define TF_GELU_TCLAMP (\S+)f\n", text).group(1))
    return np.array(coef, np.float32), clamp


def test_committed_coefficients_within_one_ulp_on_every_fp16_input():
    special = pytest.importorskip("scipy.special")
    sys.path.insert(0, CSRC)
    try:
        import gen_gelu_poly as gen
    finally:
        sys.path.remove(CSRC)
    p, clamp = _header_coefficients()
    assert clamp == gen.T_CLAMP
    worst, frac = gen.check(p)
    assert worst <= 1
    assert frac < 0.01


def test_gelu_closed_forms_at_the_ends():
    special = pytest.importorskip("scipy.special")
    sys.path.insert(0, CSRC)
    try:
        import gen_gelu_poly as gen
    finally:
        sys.path.remove(CSRC)
    p, _ = _header_coefficients()
    s = np.float32([0.0, 8.0, 20.0, 1000.0, -8.0, -20.0, -1000.0])
    y = gen.gelu_fp32(s, p).astype(np.float64)
    assert y[0] == 0.0                                  # GELU(0) = 0
    assert np.all(np.abs(y[1:4] - s[1:4]) <= 1e-6 * s[1:4])   # s * Phi(s) -> s
    assert np.all(np.abs(y[4:]) < 6e-8)                 # below the smallest fp16 subnormal
    # Phi(-s) = 1 - Phi(s): GELU(s) - GELU(-s) = s, at points inside the fit range
    t = np.float32([0.25, 0.5, 1.0, 2.0, 3.0])
    d = gen.gelu_fp32(t, p).astype(np.float64) - gen.gelu_fp32(-t, p).astype(np.float64)
    assert np.allclose(d, t, rtol=1e-5, atol=0)
    ref = t.astype(np.float64) * special.ndtr(t.astype(np.float64))
    assert np.allclose(gen.gelu_fp32(t, p).astype(np.float64), ref, rtol=3e-5, atol=0)
