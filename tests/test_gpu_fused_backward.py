"""The one-pass backward (``uaa_attn_bwd_fused``: dK, dV and dQ from one K/V-major
kernel, dQ added into an fp32 accumulator by reductions) against the fp64 oracle,
through the C ABI.

The same cases as the split backward's parity tests: ragged tiles, a single
token, prefix, random and tile-hole key masks, a fully masked batch, both head
sizes, and the layout, 1k DiT and masked workloads.  dK and dV do not depend on
the order of the dQ reductions, so they are bit-for-bit reproducible; dQ is
compared against the oracle (and against the split path within the same bar).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import ulysses_dit_attention_gb300 as uaa
from ulysses_dit_attention_gb300 import synth
from helpers import bits, compare, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _mask(kind, B, S, seed):
    g = torch.Generator().manual_seed(seed)
    if kind is None:
        return None
    if kind == "prefix":
        lens = torch.randint(S // 2, S + 1, (B,), generator=g)
        lens[0] = max(1, S // 3)
        return (torch.arange(S)[None, :] < lens[:, None]).to(torch.uint8)
    if kind == "random":
        return (torch.rand((B, S), generator=g) < 0.5).to(torch.uint8)
    if kind == "holes":  # whole 128-key tiles masked between attended ones, and one batch all masked
        m = (torch.rand((B, S), generator=g) < 0.6).to(torch.uint8)
        m[:, 128:256] = 0
        m[:, 384:512] = 0
        m[-1] = 0
        return m
    raise ValueError(kind)


def _check(inp, mask, scale, label):
    q, k, v, do = (inp[n].to(DEV) for n in ("q", "k", "v", "do"))
    m = None if mask is None else mask.to(DEV)
    o, lse = uaa.attn_fwd(q, k, v, m, scale)
    dq, dk, dv = uaa.attn_bwd(q, k, v, o, do, lse, m, scale, fused=True)
    uaa.check_device_status()
    mm = None if mask is None else mask.numpy().astype(bool)
    qq, kk, vv, dd = (f64(inp[n]) for n in ("q", "k", "v", "do"))
    rdq, rdk, rdv = oracle.attn_bwd(qq, kk, vv, dd, mm, scale)
    compare(f"{label} fused dQ", f64(dq), rdq, "dq")
    compare(f"{label} fused dK", f64(dk), rdk, "dk")
    compare(f"{label} fused dV", f64(dv), rdv, "dv")
    if mm is not None:
        for b in range(mm.shape[0]):
            assert (f64(dk)[b, ~mm[b]] == 0).all() and (f64(dv)[b, ~mm[b]] == 0).all()
    return q, k, v, do, m, o, lse, (dq, dk, dv)


CASES = [
    (2, 16, 16, 64, None),
    (1, 1, 1, 64, None),
    (1, 127, 2, 128, None),
    (2, 129, 3, 64, "prefix"),
    (1, 300, 2, 128, "random"),
    (3, 640, 2, 128, "holes"),
    (3, 640, 2, 64, "holes"),
    (1, 1000, 3, 128, None),
]


@pytest.mark.parametrize("B,S,H,D,kind", CASES)
def test_fused_backward_matches_the_oracle(B, S, H, D, kind):
    inp = synth.draw(B, S, H, D, seed=500 + S + D)
    _check(inp, _mask(kind, B, S, S + D), 1.0 / math.sqrt(D), f"B{B} S{S} H{H} D{D} {kind}")


@pytest.mark.parametrize("name", ["layout_b2_s16_h16_d64", "dit_b2_s1024_h24_d64", "mask_b4_s4096_h24_d128"])
def test_fused_backward_workloads(name):
    w = synth.workload(name)
    inp = synth.make(w)
    if w.H > 8:  # heads are independent: the oracle evaluates a subset, the GPU runs all
        q, k, v, do = (inp[n].to(DEV) for n in ("q", "k", "v", "do"))
        m = None if inp["mask"] is None else inp["mask"].to(DEV)
        o, lse = uaa.attn_fwd(q, k, v, m, w.scale)
        dq, dk, dv = uaa.attn_bwd(q, k, v, o, do, lse, m, w.scale, fused=True)
        uaa.check_device_status()
        heads = [0, w.H // 2, w.H - 1]
        qq, kk, vv, dd = (f64(inp[n])[:, :, heads] for n in ("q", "k", "v", "do"))
        mm = None if inp["mask"] is None else inp["mask"].numpy().astype(bool)
        rdq, rdk, rdv = oracle.attn_bwd(qq, kk, vv, dd, mm, w.scale)
        compare(f"{name} fused dQ", f64(dq)[:, :, heads], rdq, "dq")
        compare(f"{name} fused dK", f64(dk)[:, :, heads], rdk, "dk")
        compare(f"{name} fused dV", f64(dv)[:, :, heads], rdv, "dv")
    else:
        _check(inp, inp["mask"], w.scale, name)


@pytest.mark.parametrize("D", [64, 128])
def test_fused_backward_dk_dv_reproducible_dq_close_to_split(D):
    inp = synth.draw(2, 900, 3, D, seed=77 + D, masked=True)
    q, k, v, do, m, o, lse, (dq, dk, dv) = _check(inp, inp["mask"], 1 / math.sqrt(D), f"repro D{D}")
    dq2, dk2, dv2 = uaa.attn_bwd(q, k, v, o, do, lse, m, 1 / math.sqrt(D), fused=True)
    assert np.array_equal(bits(dk2), bits(dk)) and np.array_equal(bits(dv2), bits(dv))
    sq, sk, sv = uaa.attn_bwd(q, k, v, o, do, lse, m, 1 / math.sqrt(D))
    uaa.check_device_status()
    compare("fused vs split dQ", f64(dq2), f64(sq), "dq")
    compare("fused vs split dK", f64(dk), f64(sk), "dk")
    compare("fused vs split dV", f64(dv), f64(sv), "dv")
