"""Tensors past 2^31 elements: every kernel must address them with 64-bit offsets.

Each case has 2.2-2.3e9 elements per tensor (4.5 GB in bf16), drawn on the device
by the seeded generator of the input module:

* many short problems, B = 640, S = 200 (two tiles, the second ragged), H = 136 at
  D = 128 (272 at D = 64), with a key-padding mask: (b, h) problems are independent,
  so the oracle checks whole problems -- O, LSE, dQ, dK, dV -- at the start, in the
  middle and at the very end of the tensors, where element offsets exceed 2^31;
* one long sequence, B = 1, S = 131072, H = 136 at D = 128 (272 at D = 64): the
  oracle checks O, LSE and dQ on query-row blocks at both ends of the sequence for
  the first and the last head (each row against all keys); dK and dV, which need
  every query per key, are checked through the identities sum_j dV_j = sum_i dO_i
  and sum_j dK_j = 0 and through buffers filled with NaN before the call (every row
  must be written);
* the Ulysses re-layouts of four uneven shards of such a sequence: seq->head must
  equal plain slicing of the concatenated sequence and head->seq must restore the
  shards, bit for bit;
* the Ulysses step with the exchanges fused into the attention kernels on those
  shards (one tensor map per shard): O, LSE and dQ rows at the ends of the first
  and the last shard, first and last head, against the oracle on the whole
  sequence, and every row of the output shards written.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import ulysses_dit_attention_gb300 as uaa
from ulysses_dit_attention_gb300 import synth
from helpers import compare, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _release():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("D", [128, 64])
def test_many_problems_past_2_31_elements(D):
    B, S, H = 640, 200, 136 * 128 // D
    assert B * S * H * D > 2 ** 31
    inp = synth.draw_device(B, S, H, D, seed=31 + D, device=DEV)
    q, k, v, do = (inp[n] for n in ("q", "k", "v", "do"))
    g = torch.Generator().manual_seed(31)
    lens = torch.randint(1, S + 1, (B,), generator=g)
    mask = (torch.arange(S)[None, :] < lens[:, None]).to(torch.uint8)
    scale = 1.0 / math.sqrt(D)
    o, lse = uaa.attn_fwd(q, k, v, mask.to(DEV), scale)
    dq, dk, dv = uaa.attn_bwd(q, k, v, o, do, lse, mask.to(DEV), scale)
    uaa.check_device_status()
    for b, h in ((0, 0), (B // 2, 77), (B - 1, H - 1), (B - 1, 0)):
        sl = lambda t: f64(t[b:b + 1, :, h:h + 1])  # noqa: E731
        qq, kk, vv, dd = sl(q), sl(k), sl(v), sl(do)
        m = mask[b:b + 1].numpy().astype(bool)
        ro, rl = oracle.attn_fwd(qq, kk, vv, m, scale)
        rdq, rdk, rdv = oracle.attn_bwd(qq, kk, vv, dd, m, scale)
        label = f"b={b} h={h}"
        compare(f"{label} O", sl(o), ro, "o")
        compare(f"{label} LSE", f64(lse[b:b + 1, h:h + 1]), rl, "lse")
        compare(f"{label} dQ", sl(dq), rdq, "dq")
        compare(f"{label} dK", sl(dk), rdk, "dk")
        compare(f"{label} dV", sl(dv), rdv, "dv")
    del inp, q, k, v, do, o, lse, dq, dk, dv
    _release()


@pytest.mark.parametrize("D", [128, 64])
def test_long_sequence_past_2_31_elements(D):
    B, S, H = 1, 131072, 136 * 128 // D
    assert B * S * H * D > 2 ** 31
    inp = synth.draw_device(B, S, H, D, seed=37 + D, device=DEV)
    q, k, v, do = (inp[n] for n in ("q", "k", "v", "do"))
    scale = 1.0 / math.sqrt(D)
    o, lse = uaa.attn_fwd(q, k, v, None, scale)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    uaa.attn_bwd(q, k, v, o, do, lse, None, scale, dq=dq, dk=dk, dv=dv)
    uaa.check_device_status()
    # exact rows at both ends of the sequence, first and last head, against all keys
    for h in (0, H - 1):
        kk, vv = f64(k[:, :, h:h + 1]), f64(v[:, :, h:h + 1])
        for r0 in (0, S - 128):
            qq, dd = f64(q[:, r0:r0 + 128, h:h + 1]), f64(do[:, r0:r0 + 128, h:h + 1])
            ro, rl = oracle.attn_fwd(qq, kk, vv, None, scale)
            rdq, _, _ = oracle.attn_bwd(qq, kk, vv, dd, None, scale)
            label = f"h={h} rows {r0}..{r0 + 127}"
            compare(f"{label} O", f64(o[:, r0:r0 + 128, h:h + 1]), ro, "o")
            compare(f"{label} LSE", f64(lse[:, h:h + 1, r0:r0 + 128]), rl, "lse")
            compare(f"{label} dQ", f64(dq[:, r0:r0 + 128, h:h + 1]), rdq, "dq")
    # every row of every gradient was written
    for name, t in (("dQ", dq), ("dK", dk), ("dV", dv)):
        assert bool(torch.isfinite(t).all()), f"{name}: rows left unwritten"
    # Identities over all keys, per head and column: the rows of P sum to one, so
    # sum_j dV_j = sum_i dO_i, and the rows of dS sum to zero, so sum_j dK_j = 0.  The fp32
    # accumulation of dV over 131072 queries in the tensor core shrinks it systematically
    # by ~1e-4 (measured 1.1e-5 at S = 4096 growing to 1.4e-4 at S = 131072, with dV at
    # S = 4096 within 2.4e-3 of the oracle and biased by 8e-6), so both are held to 1e-3 of
    # their scale here; a query tile left out of the backward moves sum_j dV_j by percents.
    # (Key rows written in the wrong place leave rows unwritten, checked above; the exact
    # per-problem checks of the large-batch test cover the key side at large offsets.)
    got = dv.float().sum(dim=1).double()
    want = do.float().sum(dim=1).double()
    rel = float((got - want).abs().max() / want.abs().max())
    assert rel <= 1e-3, f"sum_j dV_j vs sum_i dO_i: relative {rel:.3e}"
    dk_sum = float(dk.float().sum(dim=1).abs().max())
    dk_abs = float(dk.float().abs().sum(dim=1).max())
    assert dk_sum <= 1e-3 * dk_abs, f"sum_j dK_j = {dk_sum:.3e} against sum_j |dK_j| = {dk_abs:.3e}"
    del inp, q, k, v, do, o, lse, dq, dk, dv
    _release()


def test_relayouts_past_2_31_elements():
    lens, B, H, D = [32770, 32768, 32767, 32767], 1, 136, 128
    P, cap, N = len(lens), max(lens), sum(lens)
    assert P * B * cap * H * D > 2 ** 31
    g = torch.Generator(device=DEV).manual_seed(41)
    x = torch.randint(-30000, 30000, (P, B, cap, H, D), generator=g, device=DEV, dtype=torch.int16)
    x = x.view(torch.bfloat16)  # arbitrary bit patterns: the re-layouts move bytes
    y = uaa.seq_to_head(x, lens)
    uaa.check_device_status()
    Hg = H // P
    assert y.shape == (P, B, N, Hg, D)
    off = 0
    for p, L in enumerate(lens):
        for grp in (0, P - 1):
            want = x[p, :, :L, grp * Hg:(grp + 1) * Hg].view(torch.int16)
            assert torch.equal(y[grp, :, off:off + L].view(torch.int16), want), f"shard {p} group {grp}"
        off += L
    back = torch.full_like(x, float("nan"))
    uaa.head_to_seq(y, lens, cap, out=back)
    uaa.check_device_status()
    for p, L in enumerate(lens):
        assert torch.equal(back[p, :, :L].view(torch.int16), x[p, :, :L].view(torch.int16)), f"shard {p}"
        assert bool((back[p, :, L:].view(torch.int16) == 0).all()), f"padding rows of shard {p}"
    del x, y, back
    _release()


def test_fused_ulysses_past_2_31_elements():
    lens, B, H, D = [32770, 32768, 32767, 32767], 1, 136, 128
    P, cap, N = len(lens), max(lens), sum(lens)
    assert P * B * cap * H * D > 2 ** 31
    inp = synth.draw_device(P * B, cap, H, D, seed=43, device=DEV)  # (P*B, cap, H, D) = the shards
    sh = {n: inp[n].view(P, B, cap, H, D) for n in ("q", "k", "v", "do")}
    scale = 1.0 / math.sqrt(D)
    o_sh, lse = uaa.ulysses_attn_fwd(sh["q"], sh["k"], sh["v"], lens, None, scale)
    dq, dk, dv = (torch.full_like(sh["q"], float("nan")) for _ in range(3))
    uaa.ulysses_attn_bwd(sh["q"], sh["k"], sh["v"], o_sh, sh["do"], lse, lens, None, scale, dq=dq, dk=dk, dv=dv)
    uaa.check_device_status()
    offs = np.concatenate([[0], np.cumsum(lens)])
    for t, name in ((o_sh, "O"), (dq, "dQ"), (dk, "dK"), (dv, "dV")):
        for p, L in enumerate(lens):
            assert bool(torch.isfinite(t[p, :, :L]).all()), f"{name}: rows of shard {p} left unwritten"
    for h in (0, H - 1):
        # the whole sequence of head h: the shards' valid rows in order
        full = {n: torch.cat([sh[n][p, :, :L, h:h + 1] for p, L in enumerate(lens)], dim=1) for n in ("q", "k", "v", "do")}
        kk, vv = f64(full["k"]), f64(full["v"])
        for p, r0 in ((0, 0), (P - 1, lens[-1] - 128)):
            n0 = int(offs[p]) + r0
            qq, dd = f64(full["q"][:, n0:n0 + 128]), f64(full["do"][:, n0:n0 + 128])
            ro, rl = oracle.attn_fwd(qq, kk, vv, None, scale)
            rdq, _, _ = oracle.attn_bwd(qq, kk, vv, dd, None, scale)
            label = f"h={h} shard {p} rows {r0}..{r0 + 127}"
            compare(f"{label} O", f64(o_sh[p, :, r0:r0 + 128, h:h + 1]), ro, "o")
            compare(f"{label} LSE", f64(lse[:, h:h + 1, n0:n0 + 128]), rl, "lse")
            compare(f"{label} dQ", f64(dq[p, :, r0:r0 + 128, h:h + 1]), rdq, "dq")
        del full
    del inp, sh, o_sh, lse, dq, dk, dv
    _release()
