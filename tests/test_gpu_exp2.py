"""The forward's FMA-pipe exponential, evaluated by the device code itself.

One column pair of P in eight takes 2^x from ``exp2_fma2`` (range reduction, a
cubic fitted by ulysses_dit_attention_gb300/exp2_fit.py, 2^n in the exponent
field) instead of the special-function unit.  ``uaa_debug_exp2_fma2`` runs that
device function over an array; its results must be within 1e-4 relative of 2^x in
float64 and of CUDA's own exp2f (torch.exp2 on the device) over the range the
softmax uses, agree with the float32 model of the same steps in the fit script to
an ulp, and give exactly 0 at and below x = -127 and for -inf.
"""
import numpy as np
import pytest
import torch

import ulysses_dit_attention_gb300 as uaa
from ulysses_dit_attention_gb300 import exp2_fit

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _inputs():
    g = torch.Generator().manual_seed(7)
    grid = torch.linspace(-125.0, 8.0, 1 << 20, dtype=torch.float32)
    rand = torch.rand(1 << 20, generator=g, dtype=torch.float32) * 133.0 - 125.0
    near_int = torch.arange(-125, 9, dtype=torch.float32).repeat_interleave(8) + torch.tensor(
        [-0.5, -0.4999, -1e-6, 0.0, 1e-6, 0.25, 0.4999, 0.5]).repeat(134)  # rounding boundaries
    return torch.cat([grid, rand, near_int])


def test_exp2_fma2_against_float64_and_exp2f():
    x = _inputs()
    if x.numel() % 2:
        x = torch.cat([x, torch.zeros(1)])
    y = uaa.debug_exp2_fma2(x.to(DEV))
    ref_f = torch.exp2(x.to(DEV))  # CUDA's exp2f
    uaa.check_device_status()
    xs, ys, rf = x.numpy().astype(np.float64), y.cpu().numpy().astype(np.float64), ref_f.cpu().numpy().astype(np.float64)
    ref = np.exp2(xs)
    rel64 = np.abs(ys - ref) / ref
    relf = np.abs(ys - rf) / rf
    assert rel64.max() < 1e-4, f"against 2^x in float64: {rel64.max():.3e} at x = {xs[rel64.argmax()]}"
    assert relf.max() < 1e-4, f"against exp2f: {relf.max():.3e} at x = {xs[relf.argmax()]}"
    # the device evaluates the fit script's float32 model of the same steps (to an ulp: the
    # model's fused multiply-adds round through float64 first)
    model = exp2_fit.eval_float32(exp2_fit.as_float32(exp2_fit.fit()), x.numpy()).astype(np.float64)
    assert (np.abs(ys - model) <= 2.0 ** -22 * np.abs(model)).all()


def test_exp2_fma2_special_values():
    x = torch.tensor([-float("inf"), -1000.0, -200.0, -127.0, -127.4, 0.0, 1.0, 8.0], dtype=torch.float32)
    y = uaa.debug_exp2_fma2(x.to(DEV)).cpu()
    uaa.check_device_status()
    assert (y[:5] == 0).all(), y[:5]
    assert torch.allclose(y[5:], torch.tensor([1.0, 2.0, 256.0]), rtol=1e-4, atol=0)
    with pytest.raises(ValueError):
        uaa.debug_exp2_fma2(torch.zeros(3, device=DEV))
