"""Coefficients of the cubic that the kernels use for 2^f on [-1/2, 1/2].

The attention kernels compute part of their exponentials on the FMA pipe
instead of the special-function unit: x = n + f with n = rint(x) and
|f| <= 1/2, 2^f by the cubic c0 + c1 f + c2 f^2 + c3 f^3 below, 2^n by
writing n + 127 into the exponent field.  The cubic is a near-minimax fit in
relative error, computed here by Lawson's iteratively reweighted least squares
on a dense grid (plain numpy, float64).  Its relative error (about 9e-5) is far
below the bf16 rounding (2^-9) that P receives before the P V product.

``python -m ulysses_dit_attention_gb300.exp2_fit`` prints the coefficients as
float32 literals and the maximum relative error of the float32 evaluation.
"""
from __future__ import annotations

import numpy as np

DEGREE = 3


def fit(degree: int = DEGREE, iters: int = 400, npts: int = 4001) -> np.ndarray:
    """Near-minimax coefficients (c0 .. c_degree) of 2^f in relative error on [-1/2, 1/2]."""
    f = np.linspace(-0.5, 0.5, npts)
    y = np.exp2(f)
    a = np.vander(f, degree + 1, increasing=True) / y[:, None]  # relative-error rows
    w = np.full(npts, 1.0 / npts)
    c = None
    for _ in range(iters):
        sw = np.sqrt(w)
        c, *_ = np.linalg.lstsq(a * sw[:, None], np.ones(npts) * sw, rcond=None)
        err = np.abs(a @ c - 1.0)
        w = w * err
        w /= w.sum()
    return c


def as_float32(c: np.ndarray) -> np.ndarray:
    return np.asarray(c, dtype=np.float32)


def eval_float32(c32: np.ndarray, x: np.ndarray) -> np.ndarray:
    """The device sequence in float32: clamp, round by the 1.5*2^23 shift, Horner by fused
    multiply-adds (each rounded once to float32), exponent field, one product."""
    x = np.maximum(np.asarray(x, dtype=np.float32), np.float32(-127.0))
    shift = np.float32(12582912.0)
    t = (x + shift).astype(np.float32)
    n = (t - shift).astype(np.float32)
    f = (x - n).astype(np.float32)
    p = np.full_like(f, c32[-1])
    for k in range(len(c32) - 2, -1, -1):
        p = (p.astype(np.float64) * f.astype(np.float64) + np.float64(c32[k])).astype(np.float32)
    bits = ((t.view(np.uint32).astype(np.uint64) << 23) + 0x3F800000) & 0xFFFFFFFF
    scale = bits.astype(np.uint32).view(np.float32)
    return (p * scale).astype(np.float32)


def max_rel_error(c32: np.ndarray, lo: float = -30.0, hi: float = 8.0, npts: int = 200001) -> float:
    x = np.linspace(lo, hi, npts).astype(np.float32)
    ref = np.exp2(x.astype(np.float64))
    return float(np.max(np.abs(eval_float32(c32, x).astype(np.float64) - ref) / ref))


if __name__ == "__main__":
    c32 = as_float32(fit())
    for k, v in enumerate(c32):
        print(f"c{k} = {float(v):.9e}f  (bits 0x{np.float32(v).view(np.uint32):08x})")
    print(f"max relative error of the float32 evaluation on [-30, 8]: {max_rel_error(c32):.3e}")
