"""The cubic behind the kernels' FMA-pipe exponentials (exp2_fma2).

The coefficients compiled into the CUDA header must be the ones the fit in
ulysses_dit_attention_gb300/exp2_fit.py produces, and the float32 evaluation of
the device sequence (clamp, rounding shift, Horner by fused multiply-adds,
exponent field) must stay within 1e-4 relative error of 2^x over the range the
softmax uses, give exactly 0 for -inf and for x <= -127, and 1 at x = 0 to
within the same bound.  No GPU: numpy only.
"""
import os
import re

import numpy as np

from ulysses_dit_attention_gb300 import exp2_fit

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "ulysses_dit_attention_gb300", "csrc", "uaa_common.cuh")


def _header_coefficients():
    src = open(HEADER).read()
    body = src[src.index("float2 exp2_fma2("):]
    body = body[: body.index("}")]
    found = dict(re.findall(r"\b(c[0-3]) = ([-+0-9.eE]+)f", body))
    return np.array([float(found[f"c{k}"]) for k in range(4)], dtype=np.float32)


def test_header_coefficients_are_the_fit():
    fitted = exp2_fit.as_float32(exp2_fit.fit())
    header = _header_coefficients()
    # printed with 10 significant digits: the same float32 values
    assert np.array_equal(fitted, header), (fitted, header)


def test_relative_error_bound():
    c32 = _header_coefficients()
    assert exp2_fit.max_rel_error(c32, -30.0, 8.0) < 1e-4
    # well below half an ulp of bf16, the precision P is rounded to
    assert exp2_fit.max_rel_error(c32, -30.0, 8.0) < 2.0 ** -9 / 10


def test_special_values():
    c32 = _header_coefficients()
    x = np.array([-np.inf, -1000.0, -127.0, -126.6, 0.0, 1.0, 8.0], dtype=np.float32)
    y = exp2_fit.eval_float32(c32, x)
    assert y[0] == 0.0 and y[1] == 0.0 and y[2] == 0.0 and y[3] == 0.0
    assert abs(y[4] - 1.0) < 1e-4
    assert abs(y[5] / 2.0 - 1.0) < 1e-4
    assert abs(y[6] / 256.0 - 1.0) < 1e-4


def test_integer_arguments_are_exact_powers_times_c0():
    # at f = 0 the cubic returns c0, so 2^n comes out as c0 * 2^n exactly
    c32 = _header_coefficients()
    n = np.arange(-120, 9, dtype=np.float32)
    y = exp2_fit.eval_float32(c32, n)
    assert np.array_equal(y, (c32[0] * np.exp2(n.astype(np.float64))).astype(np.float32))
