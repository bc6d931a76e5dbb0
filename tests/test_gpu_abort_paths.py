"""The attention kernels' abort paths on the GPU, made to run without any fault.

Every wait of a kernel role for another role's progress is bounded.  The
diagnostic ``uaa_debug_drop_load(n)`` makes each producer skip its n-th ring
load: nothing ever fills that buffer (no copy is issued at all), so the waits
for it run out after the wait bound (set to 20 ms here).  The kernel then
records a timeout, every role leaves its loops -- the forward's softmax and
issuer warps keep meeting at every named barrier of the schedule -- the copies
and MMAs already issued are waited for, TMEM is released and the kernel
returns.  Each test runs one or two work items per kernel, checks that
``uaa_check_device_status`` reports ``UAA_ERR_TIMEOUT``, and that the next call
(ordinary settings, issued before the status was read) gives the same bits as
a call before the failure: the give-up is scoped to the call that failed.
"""
import math

import numpy as np
import pytest
import torch

import ulysses_dit_attention_gb300 as uaa
from ulysses_dit_attention_gb300 import synth
from helpers import bits

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _inputs(S, D, masked):
    inp = synth.draw(1, S, 1, D, seed=90 + S + D, masked=False)
    q, k, v, do = (inp[n].to(DEV) for n in ("q", "k", "v", "do"))
    mask = None
    if masked:
        mask = torch.zeros((1, S), dtype=torch.uint8)
        mask[0, : S // 2 + 1] = 1
        mask = mask.to(DEV)
    return q, k, v, do, mask


class dropped_load:
    """Within the block, producers skip their n-th ring load and waits give up after 20 ms."""

    def __init__(self, n):
        self.n = n

    def __enter__(self):
        uaa.set_wait_timeout_ms(20)
        uaa.debug_drop_load(self.n)

    def __exit__(self, *a):
        uaa.debug_drop_load(-1)
        uaa.set_wait_timeout_ms(0)


def _expect_timeout():
    with pytest.raises(uaa.UAAError) as e:
        uaa.check_device_status()
    assert e.value.status == -5, str(e.value)
    uaa.check_device_status()  # read and cleared


# S = 256: one forward item (a pair of query tiles) over two key tiles, whose ring loads
# are K0 V0 K1 V1; load 3 (V1) never arrives, mid-item, after the issuer has started.
@pytest.mark.parametrize("S,D,masked,n", [(256, 128, False, 3), (256, 64, True, 3), (256, 128, False, 0)])
def test_forward_gives_up_and_the_next_call_is_correct(S, D, masked, n):
    q, k, v, do, mask = _inputs(S, D, masked)
    scale = 1.0 / math.sqrt(D)
    ref = uaa.attn_fwd(q, k, v, mask, scale)
    uaa.check_device_status()
    with dropped_load(n):
        uaa.attn_fwd(q, k, v, mask, scale)
    # the next call is enqueued before the status is read
    again = uaa.attn_fwd(q, k, v, mask, scale)
    torch.cuda.synchronize()
    _expect_timeout()
    for a, b in zip(again, ref):
        assert np.array_equal(bits(a), bits(b))


# S = 256: the dK/dV kernel has two items (key tiles) of two query-tile loads each (n = 0, 1);
# the dQ kernel two items (query tiles) of four K/V loads each (n = 0..3).  n = 3 starves the
# dQ kernel alone; n = 1 starves the dK/dV kernel, and the dQ kernel of the same call then
# stops at its first wait that is not already satisfied.
@pytest.mark.parametrize("S,D,masked,n", [(256, 128, False, 3), (256, 128, False, 1), (256, 64, True, 1)])
def test_backward_gives_up_and_the_next_call_is_correct(S, D, masked, n):
    q, k, v, do, mask = _inputs(S, D, masked)
    scale = 1.0 / math.sqrt(D)
    o, lse = uaa.attn_fwd(q, k, v, mask, scale)
    ref = uaa.attn_bwd(q, k, v, o, do, lse, mask, scale)
    uaa.check_device_status()
    with dropped_load(n):
        uaa.attn_bwd(q, k, v, o, do, lse, mask, scale)
    again = uaa.attn_bwd(q, k, v, o, do, lse, mask, scale)
    torch.cuda.synchronize()
    _expect_timeout()
    for a, b in zip(again, ref):
        assert np.array_equal(bits(a), bits(b))


def test_fused_ulysses_gives_up_and_the_next_call_is_correct():
    lens, cap = (100, 60), 100
    inp = synth.draw(1, sum(lens), 2, 128, seed=5)
    sh = {n: synth.pad_shards(inp[n], lens, cap).to(DEV) for n in ("q", "k", "v", "do")}
    o, lse = uaa.ulysses_attn_fwd(sh["q"], sh["k"], sh["v"], lens)
    ref = uaa.ulysses_attn_bwd(sh["q"], sh["k"], sh["v"], o, sh["do"], lse, lens)
    uaa.check_device_status()
    with dropped_load(1):
        uaa.ulysses_attn_fwd(sh["q"], sh["k"], sh["v"], lens)
        uaa.ulysses_attn_bwd(sh["q"], sh["k"], sh["v"], o, sh["do"], lse, lens)
    o3, lse3 = uaa.ulysses_attn_fwd(sh["q"], sh["k"], sh["v"], lens)
    again = uaa.ulysses_attn_bwd(sh["q"], sh["k"], sh["v"], o3, sh["do"], lse3, lens)
    torch.cuda.synchronize()
    _expect_timeout()
    assert np.array_equal(bits(o3), bits(o)) and np.array_equal(bits(lse3), bits(lse))
    for a, b in zip(again, ref):
        assert np.array_equal(bits(a), bits(b))
