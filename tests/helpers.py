"""Shared helpers of the GPU parity tests: conversions and the acceptance bar.

Acceptance bar against the fp64 oracle on the same bf16-rounded inputs:
max-abs error <= 1e-2 on O, <= 1e-3 on LSE, <= 2e-2 on dQ/dK/dV, and relative
Frobenius error ||x - ref||_F / ||ref||_F <= 1e-2 on every float output.
Re-layouts and the mask assembly are compared bit for bit.
"""
import numpy as np
import torch

TOL_MAX_ABS = {"o": 1e-2, "lse": 1e-3, "dq": 2e-2, "dk": 2e-2, "dv": 2e-2}
TOL_REL_FRO = 1e-2


def f64(t):
    """bf16/fp32 torch tensor (any device) -> float64 numpy array (exact)."""
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)


def bits(t):
    """Raw bit pattern of a torch tensor as a numpy integer array."""
    t = t.detach().cpu().contiguous()
    if t.element_size() == 2:
        return t.view(torch.int16).numpy()
    if t.element_size() == 4:
        return t.view(torch.int32).numpy()
    return t.view(torch.uint8).numpy()


def compare(name, got, ref, kind=None, magnitude_scaled=False):
    """Assert the acceptance bar; returns (max_abs, rel_fro).

    The max-abs bars are stated for the workloads (N(0,1) inputs, scale 1/sqrt(D)),
    whose outputs are O(1).  With ``magnitude_scaled`` (used for a non-default
    softmax scale or a single key, where outputs grow to several units) the
    max-abs bar is multiplied by max(1, max|ref|): the same relative accuracy at
    the tensor's magnitude.  A bar per element (the stated bar plus a bf16 ULP of
    that element) does not fit: the error of an element comes from the bf16
    rounding of the contraction's operands (P and dS), which can be much larger
    than the element itself after cancellation -- at scale 0.37 a dQ element of
    1.2 carries an error of 0.039 from dS entries of ~10.  The relative
    Frobenius bar is unchanged.
    """
    kind = kind or name
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    fin = np.isfinite(ref)
    # non-finite reference values (LSE = -inf of a fully masked row) must match exactly
    assert np.array_equal(got[~fin], ref[~fin]), f"{name}: non-finite entries differ"
    assert np.isfinite(got[fin]).all(), f"{name}: non-finite GPU values"
    err = np.abs(got[fin] - ref[fin])
    max_abs = float(err.max()) if err.size else 0.0
    nrm = float(np.linalg.norm(ref[fin]))
    rel = float(np.linalg.norm(got[fin] - ref[fin]) / nrm) if nrm > 0 else float(np.linalg.norm(got[fin]))
    bar = TOL_MAX_ABS[kind]
    if magnitude_scaled and fin.any():
        bar *= max(1.0, float(np.abs(ref[fin]).max()))
    assert max_abs <= bar, f"{name}: max-abs {max_abs:.3e} > {bar:.3e}"
    if nrm > 0:
        assert rel <= TOL_REL_FRO, f"{name}: rel-Frobenius {rel:.3e} > {TOL_REL_FRO}"
    return max_abs, rel
