"""The allocation-free backward entry point, through the C ABI.

``uaa_attn_bwd_noalloc`` serves callers that cannot allocate device memory when
they run the backward (allocator callbacks, plugins restricted to the stream
they were handed, runtimes with pre-planned allocations): it uses a scratch
array built into the library instead of a caller-provided workspace.  Both
entry points run the same deterministic kernels, so its gradients must equal
those of ``uaa_attn_bwd`` (the entry point with a workspace) bit for bit, on
consecutive calls that reuse the shared array -- the second parametrised shape
runs over the scratch contents left by the first.  This file is collected last
on purpose.
"""
import ctypes
import math

import pytest
import torch

import ulysses_dit_attention_gb300 as uaa
from ulysses_dit_attention_gb300 import build as uaa_build
from ulysses_dit_attention_gb300 import synth
from helpers import compare, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc_bwd(q, k, v, o, do, lse, mask, scale):
    B, S, H, D = q.shape
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = uaa.lib().uaa_attn_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(mask), _p(dq), _p(dk),
                                        _p(dv), B, S, H, D, ctypes.c_float(scale), stream)
    assert st == 0, uaa.lib().uaa_last_error().decode()
    return dq, dk, dv


@pytest.mark.parametrize("B,S,H,D,masked", [(2, 300, 3, 128, True), (1, 1000, 4, 64, False)])
def test_noalloc_backward_matches_workspace_backward_twice(B, S, H, D, masked):
    uaa_build.build()
    inp = synth.draw(B, S, H, D, seed=77 + S, masked=masked)
    q, k, v, do = (inp[n].to(DEV) for n in ("q", "k", "v", "do"))
    mask = inp["mask"].to(DEV) if masked else None
    scale = 1.0 / math.sqrt(D)
    o, lse = uaa.attn_fwd(q, k, v, mask, scale)
    ref = uaa.attn_bwd(q, k, v, o, do, lse, mask, scale)
    uaa.check_device_status()
    for _ in range(2):  # the second call reuses the scratch the first one left behind
        got = _noalloc_bwd(q, k, v, o, do, lse, mask, scale)
        uaa.check_device_status()
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert torch.equal(g.view(torch.int16), r.view(torch.int16)), f"noalloc {name} differs"
            compare(f"noalloc {name}", f64(g), f64(r), name)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    uaa_build.build()
    L = uaa.lib()
    cap = L.uaa_attn_bwd_noalloc_max_bytes()
    assert cap == 64 << 20
    B, S, H, D = 16, 27280, 40, 128
    assert L.uaa_attn_bwd_workspace_bytes(B, S, H, D) > cap
    fake = ctypes.c_void_p(1 << 20)
    st = L.uaa_attn_bwd_noalloc(fake, fake, fake, fake, fake, fake, None, fake, fake, fake, B, S, H, D,
                                ctypes.c_float(0.088), None)
    assert st == -2
    assert "scratch" in L.uaa_last_error().decode()
