"""GPU attention forward/backward (through the C ABI) vs the fp64 oracle.

Small and ragged cases are compared element by element on every output; the
large workloads (S = 4096 masked, S = 27280) are compared exactly on sampled
heads (heads are independent, so the oracle evaluates just those heads) and on
sampled query rows; the Ulysses emulation is checked against the oracle and,
bit for bit, against the plain full-sequence path.
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


def run_gpu(inp, scale, mask):
    q, k, v, do = (inp[n].to(DEV) for n in ("q", "k", "v", "do"))
    m = None if mask is None else mask.to(DEV)
    o, lse = uaa.attn_fwd(q, k, v, m, scale)
    dq, dk, dv = uaa.attn_bwd(q, k, v, o, do, lse, m, scale)
    uaa.check_device_status()
    return o, lse, dq, dk, dv


def check_against_oracle(inp, mask, scale, heads=None, label="", magnitude_scaled=False):
    o, lse, dq, dk, dv = run_gpu(inp, scale, mask)
    sel = slice(None) if heads is None else list(heads)
    q, k, v, do = (f64(inp[n])[:, :, sel] for n in ("q", "k", "v", "do"))
    m = None if mask is None else mask.numpy().astype(bool)
    ro, rl = oracle.attn_fwd(q, k, v, m, scale)
    rdq, rdk, rdv = oracle.attn_bwd(q, k, v, do, m, scale)
    res = {}
    ms = magnitude_scaled
    res["o"] = compare(f"{label} O", f64(o)[:, :, sel], ro, "o", ms)
    res["lse"] = compare(f"{label} LSE", f64(lse)[:, sel], rl, "lse", ms)
    res["dq"] = compare(f"{label} dQ", f64(dq)[:, :, sel], rdq, "dq", ms)
    res["dk"] = compare(f"{label} dK", f64(dk)[:, :, sel], rdk, "dk", ms)
    res["dv"] = compare(f"{label} dV", f64(dv)[:, :, sel], rdv, "dv", ms)
    if m is not None:
        # masked keys receive exactly zero dK / dV
        dkn, dvn = f64(dk), f64(dv)
        for b in range(m.shape[0]):
            assert (dkn[b, ~m[b]] == 0).all() and (dvn[b, ~m[b]] == 0).all()
    return res


SMALL = [
    # B, S, H, D, mask kind
    (2, 16, 16, 64, None),        # layout trap: H == S
    (1, 1, 1, 64, None),          # single token
    (1, 127, 2, 128, None),       # one ragged tile
    (2, 129, 3, 64, "prefix"),    # two tiles, ragged, prefix mask
    (1, 300, 2, 128, "random"),   # three tiles, arbitrary (non-prefix) mask
    (2, 257, 2, 128, "empty_b1"), # batch 1 fully masked: O = 0, LSE = -inf, no grads
    (1, 640, 4, 64, "prefix"),    # mask ends inside a tile, whole masked tiles
]


@pytest.mark.parametrize("B,S,H,D,kind", SMALL)
def test_small_and_ragged_cases(B, S, H, D, kind):
    inp = synth.draw(B, S, H, D, seed=1000 + S + H, masked=False)
    mask = None
    g = torch.Generator().manual_seed(S)
    if kind == "prefix":
        lens = torch.randint(S // 2, S + 1, (B,), generator=g)
        lens[0] = max(1, S // 3)
        mask = (torch.arange(S)[None, :] < lens[:, None]).to(torch.uint8)
    elif kind == "random":
        mask = (torch.rand((B, S), generator=g) < 0.5).to(torch.uint8)
    elif kind == "empty_b1":
        mask = torch.ones((B, S), dtype=torch.uint8)
        mask[1] = 0
        mask[0, 200:] = 0
    check_against_oracle(inp, mask, 1.0 / math.sqrt(D), label=f"B{B} S{S} H{H} D{D} {kind}")
    if kind == "empty_b1":
        o, lse, dq, dk, dv = run_gpu(inp, 1.0 / math.sqrt(D), mask)
        assert (f64(o)[1] == 0).all() and np.isneginf(f64(lse)[1]).all()
        assert (f64(dq)[1] == 0).all() and (f64(dk)[1] == 0).all() and (f64(dv)[1] == 0).all()


def tile_pattern_mask(B, S, patterns, seed):
    """Key mask built per 128-key tile: pattern character 'x' = every key of the tile masked,
    'p' = a random ~60 % of its keys attended, 'a' = all attended.  One pattern per batch."""
    g = torch.Generator().manual_seed(seed)
    m = torch.zeros((B, S), dtype=torch.uint8)
    for b, pat in enumerate(patterns):
        for t, c in enumerate(pat):
            lo, hi = 128 * t, min(S, 128 * (t + 1))
            if c == "a":
                m[b, lo:hi] = 1
            elif c == "p":
                m[b, lo:hi] = (torch.rand(hi - lo, generator=g) < 0.6).to(torch.uint8)
    return m


@pytest.mark.parametrize("D", [64, 128])
def test_fully_masked_key_tiles_between_attended_ones(D):
    """Key tiles 1 and 3 hold no attended key while tiles 0, 2 and 4 are partly attended:
    the forward skips the empty tiles and the dK/dV and dQ kernels walk around them, each
    role on its own, so they must agree on which tiles exist.  A second batch has a
    different pattern (its own tile count), a third none attended at all."""
    B, S, H = 3, 640, 2
    inp = synth.draw(B, S, H, D, seed=640 + D)
    mask = tile_pattern_mask(B, S, ["pxpxp", "xxaxp", "xxxxx"], seed=D)
    res = check_against_oracle(inp, mask, 1.0 / math.sqrt(D), label=f"interior-masked D{D}")
    o, lse, dq, dk, dv = run_gpu(inp, 1.0 / math.sqrt(D), mask)
    assert (f64(o)[2] == 0).all() and np.isneginf(f64(lse)[2]).all()
    assert (f64(dq)[2] == 0).all() and (f64(dk)[2] == 0).all() and (f64(dv)[2] == 0).all()
    for b, t in ((0, 1), (0, 3), (1, 0), (1, 1), (1, 3)):
        assert (f64(dk)[b, 128 * t:128 * (t + 1)] == 0).all() and (f64(dv)[b, 128 * t:128 * (t + 1)] == 0).all()
    assert res["o"][0] > 0  # the attended rows were compared against nonzero values


@pytest.mark.parametrize("B", [256, 260])
def test_many_mask_rows(B):
    """Up to 256 mask rows the forward and the dQ kernel tabulate each row's attended key
    tiles and skip the others; above that they visit every tile and the masked keys only get
    P = 0.  Both sides of the limit, with rows whose every key is masked (O = 0, LSE = -inf,
    no gradients: in the second mode that row goes through the softmax with no attended key)."""
    S, H, D = 300, 1, 64
    inp = synth.draw(B, S, H, D, seed=B)
    pats = ["pxp", "xxa", "xxx", "aap", "xpx"]
    mask = tile_pattern_mask(B, S, [pats[b % len(pats)] for b in range(B)], seed=B)
    check_against_oracle(inp, mask, 1.0 / math.sqrt(D), label=f"{B} mask rows")
    o, lse, dq, dk, dv = run_gpu(inp, 1.0 / math.sqrt(D), mask)
    empty = [b for b in range(B) if pats[b % len(pats)] == "xxx"]
    assert (f64(o)[empty] == 0).all() and np.isneginf(f64(lse)[empty]).all()
    assert (f64(dq)[empty] == 0).all() and (f64(dk)[empty] == 0).all() and (f64(dv)[empty] == 0).all()


def test_non_default_scale():
    # scale 0.37 (~3x 1/sqrt(64)) sharpens the softmax; gradients reach |dQ| ~ 6
    inp = synth.draw(1, 200, 2, 64, seed=7)
    check_against_oracle(inp, None, 0.37, label="scale 0.37", magnitude_scaled=True)


def test_layout_workload_full():
    w = synth.workload("layout_b2_s16_h16_d64")
    check_against_oracle(synth.make(w), None, w.scale, label=w.name)


def test_dit_1k_workload_full():
    w = synth.workload("dit_b2_s1024_h24_d64")
    check_against_oracle(synth.make(w), None, w.scale, label=w.name)


def test_mask_workload_sampled_heads():
    w = synth.workload("mask_b4_s4096_h24_d128")
    inp = synth.make(w)
    check_against_oracle(inp, inp["mask"], w.scale, heads=[0, 11, 23], label=w.name)


@pytest.mark.parametrize("D,masked", [(128, False), (64, True)])
def test_forward_and_backward_are_deterministic(D, masked):
    # no atomics anywhere: two runs give identical bits for O, LSE, dQ, dK, dV
    inp = synth.draw(2, 513, 2, D, seed=3, masked=masked)
    a = run_gpu(inp, 1 / math.sqrt(D), inp["mask"])
    b = run_gpu(inp, 1 / math.sqrt(D), inp["mask"])
    for x, y in zip(a, b):
        assert np.array_equal(bits(x), bits(y))
    assert np.isfinite(f64(a[1])).all()


@pytest.mark.parametrize("name", ["dit_b1_s27280_h40_d128"])
def test_dit_27k_workload_sampled(name):
    w = synth.workload(name)
    inp = synth.make(w)
    o, lse, dq, dk, dv = run_gpu(inp, w.scale, None)
    # one whole head, every output, exactly
    h = [w.H - 1]
    q, k, v, do = (f64(inp[n])[:, :, h] for n in ("q", "k", "v", "do"))
    ro, rl = oracle.attn_fwd(q, k, v, None, w.scale)
    rdq, rdk, rdv = oracle.attn_bwd(q, k, v, do, None, w.scale)
    compare("O", f64(o)[:, :, h], ro, "o")
    compare("LSE", f64(lse)[:, h], rl, "lse")
    compare("dQ", f64(dq)[:, :, h], rdq, "dq")
    compare("dK", f64(dk)[:, :, h], rdk, "dk")
    compare("dV", f64(dv)[:, :, h], rdv, "dv")
    # sampled query rows of two more heads: O, LSE and dQ rows are exact per row
    rows = np.array([0, 1, 127, 128, 13653, 27151, 27152, 27279])
    for hh in (0, 17):
        qs = f64(inp["q"])[:, rows][:, :, [hh]]
        dos = f64(inp["do"])[:, rows][:, :, [hh]]
        kk, vv = f64(inp["k"])[:, :, [hh]], f64(inp["v"])[:, :, [hh]]
        ro, rl = oracle.attn_fwd(qs, kk, vv, None, w.scale)
        rdq, _, _ = oracle.attn_bwd(qs, kk, vv, dos, None, w.scale)
        compare(f"O rows h{hh}", f64(o)[:, rows][:, :, [hh]], ro, "o")
        compare(f"LSE rows h{hh}", f64(lse)[:, [hh]][:, :, rows], rl, "lse")
        compare(f"dQ rows h{hh}", f64(dq)[:, rows][:, :, [hh]], rdq, "dq")


def test_ulysses_emulation_workload():
    """seq->head, attention per 10-head group, head->seq; fwd + bwd.

    The forward and all three gradients equal the full-sequence path bit for
    bit (same inputs, the head groups are exact head slices, and the kernels
    are deterministic).
    """
    w = synth.workload("ulysses_p4_n27280_h40_d128")
    inp = synth.make(w)
    lens, cap = w.shard_lens, w.cap
    sh = {n: synth.pad_shards(inp[n], lens, cap).to(DEV) for n in ("q", "k", "v", "do")}
    q_sh = sh["q"].requires_grad_(True)
    k_sh = sh["k"].requires_grad_(True)
    v_sh = sh["v"].requires_grad_(True)
    o_sh, lse_g = uaa.ulysses_attention(q_sh, k_sh, v_sh, lens, None, w.scale)
    o_sh.backward(sh["do"])
    uaa.check_device_status()
    # padding rows of every returned shard are zero
    for p, L in enumerate(lens):
        for t in (o_sh, q_sh.grad, k_sh.grad, v_sh.grad):
            assert (bits(t[p, :, L:]) == 0).all()
    # reference: the plain path on the unsharded sequence
    o, lse, dq, dk, dv = run_gpu(inp, w.scale, None)

    def unshard(t):
        return torch.cat([t[p, :, :L] for p, L in enumerate(lens)], dim=1)

    assert np.array_equal(bits(unshard(o_sh.detach())), bits(o))
    hg = w.H // w.P
    for g in range(w.P):
        assert np.array_equal(bits(lse_g[g]), bits(lse[:, g * hg:(g + 1) * hg]))
    assert np.array_equal(bits(unshard(k_sh.grad)), bits(dk))
    assert np.array_equal(bits(unshard(v_sh.grad)), bits(dv))
    assert np.array_equal(bits(unshard(q_sh.grad)), bits(dq))
    # and the oracle on one head of the last group, through the oracle's own exchange
    h = [w.H - 3]
    q, k, v, do = (f64(inp[n])[:, :, h] for n in ("q", "k", "v", "do"))
    rdq, rdk, rdv = oracle.attn_bwd(q, k, v, do, None, w.scale)
    ro, _ = oracle.attn_fwd(q, k, v, None, w.scale)
    compare("ulysses O", f64(unshard(o_sh.detach()))[:, :, h], ro, "o")
    compare("ulysses dQ", f64(unshard(q_sh.grad))[:, :, h], rdq, "dq")
    compare("ulysses dK", f64(unshard(k_sh.grad))[:, :, h], rdk, "dk")
    compare("ulysses dV", f64(unshard(v_sh.grad))[:, :, h], rdv, "dv")


CROSS = [
    # B, Sq, Sk, H, D, masked
    (2, 300, 700, 3, 128, True),    # more keys than queries, ragged tiles, key mask (B, Sk)
    (1, 1000, 257, 2, 64, False),   # more queries than keys
    (1, 128, 1, 2, 128, False),     # a single key
]


@pytest.mark.parametrize("B,Sq,Sk,H,D,masked", CROSS)
def test_cross_attention_sq_ne_sk(B, Sq, Sk, H, D, masked):
    """Separate query and key lengths ("[attention] Add Ulysses Anything backward", What does
    this PR do: query and key partition metadata are kept separately)."""
    g = torch.Generator().manual_seed(Sq * 7 + Sk)
    q = torch.randn((B, Sq, H, D), generator=g).to(torch.bfloat16)
    k, v = (torch.randn((B, Sk, H, D), generator=g).to(torch.bfloat16) for _ in range(2))
    do = torch.randn((B, Sq, H, D), generator=g).to(torch.bfloat16)
    mask = None
    if masked:
        lens = torch.randint(Sk // 2, Sk + 1, (B,), generator=g)
        mask = (torch.arange(Sk)[None, :] < lens[:, None]).to(torch.uint8)
    scale = 1.0 / np.sqrt(D)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    md = None if mask is None else mask.to(DEV)
    o, lse = uaa.attn_fwd(qd, kd, vd, md, scale)
    dq, dk, dv = uaa.attn_bwd(qd, kd, vd, o, dod, lse, md, scale)
    uaa.check_device_status()
    assert tuple(o.shape) == (B, Sq, H, D) and tuple(lse.shape) == (B, H, Sq)
    assert tuple(dq.shape) == (B, Sq, H, D) and tuple(dk.shape) == (B, Sk, H, D)
    m = None if mask is None else mask.numpy().astype(bool)
    qq, kk, vv, dd = (f64(t) for t in (q, k, v, do))
    ro, rl = oracle.attn_fwd(qq, kk, vv, m, scale)
    rdq, rdk, rdv = oracle.attn_bwd(qq, kk, vv, dd, m, scale)
    # with a single key every query puts weight 1 on it: dV is a sum of Sq rows of dO (|dV| ~ sqrt(Sq)),
    # so the absolute bar is scaled by the reference magnitude there (the same relative accuracy)
    ms = Sk == 1
    compare("cross O", f64(o), ro, "o")
    compare("cross LSE", f64(lse), rl, "lse")
    compare("cross dQ", f64(dq), rdq, "dq", ms)
    compare("cross dK", f64(dk), rdk, "dk", ms)
    compare("cross dV", f64(dv), rdv, "dv", ms)
    if m is not None:
        for b in range(B):
            assert (f64(dk)[b, ~m[b]] == 0).all() and (f64(dv)[b, ~m[b]] == 0).all()


def test_ulysses_padded_heads_equal_the_unsharded_path():
    """P = 4 does not divide H = 6: the head groups carry zero padding heads.

    Attention on a zero head is well defined (uniform weights, O = 0, zero
    gradients) and the padding heads are dropped on the way back, so the real
    heads' O, LSE and gradients equal the unsharded path bit for bit.
    """
    lens, cap = (301, 300, 257, 130), 301
    B, H, D = 2, 6, 128
    inp = synth.draw(B, sum(lens), H, D, seed=31)
    scale = 1.0 / np.sqrt(D)
    sh = {n: synth.pad_shards(inp[n], lens, cap).to(DEV) for n in ("q", "k", "v", "do")}
    q_sh = sh["q"].requires_grad_(True)
    k_sh = sh["k"].requires_grad_(True)
    v_sh = sh["v"].requires_grad_(True)
    o_sh, lse_g = uaa.ulysses_attention(q_sh, k_sh, v_sh, lens, None, scale)
    o_sh.backward(sh["do"])
    uaa.check_device_status()
    assert tuple(o_sh.shape) == (4, B, cap, H, D) and tuple(lse_g.shape) == (4, B, 2, sum(lens))
    o, lse, dq, dk, dv = run_gpu(inp, scale, None)

    def unshard(t):
        return torch.cat([t[p, :, :L] for p, L in enumerate(lens)], dim=1)

    assert np.array_equal(bits(unshard(o_sh.detach())), bits(o))
    for h in range(H):
        assert np.array_equal(bits(lse_g[h // 2][:, h % 2]), bits(lse[:, h]))
    assert np.array_equal(bits(unshard(q_sh.grad)), bits(dq))
    assert np.array_equal(bits(unshard(k_sh.grad)), bits(dk))
    assert np.array_equal(bits(unshard(v_sh.grad)), bits(dv))
    for p, L in enumerate(lens):
        for t in (o_sh, q_sh.grad, k_sh.grad, v_sh.grad):
            assert (bits(t[p, :, L:]) == 0).all()


@pytest.mark.parametrize("D,masked", [(128, True), (64, False)])
def test_grouped_launch_equals_one_call_per_group(D, masked):
    """uaa_attn_fwd_groups / uaa_attn_bwd_groups: G head groups of B sequences in one launch,
    the B mask rows shared by every group, equal G separate calls bit for bit."""
    G, B, S, H = 3, 2, 300, 2
    g = torch.Generator().manual_seed(33 + D)
    q, k, v, do = (torch.randn((G, B, S, H, D), generator=g).to(torch.bfloat16).to(DEV) for _ in range(4))
    mask = None
    if masked:
        mask = tile_pattern_mask(B, S, ["pxp", "app"], seed=3).to(DEV)
    scale = 1.0 / math.sqrt(D)
    o, lse = uaa.attn_fwd_groups(q, k, v, mask, scale)
    dq, dk, dv = uaa.attn_bwd_groups(q, k, v, o, do, lse, mask, scale)
    uaa.check_device_status()
    for gi in range(G):
        o1, l1 = uaa.attn_fwd(q[gi], k[gi], v[gi], mask, scale)
        g1 = uaa.attn_bwd(q[gi], k[gi], v[gi], o1, do[gi], l1, mask, scale)
        assert np.array_equal(bits(o[gi]), bits(o1)) and np.array_equal(bits(lse[gi]), bits(l1))
        for a, b in zip((dq, dk, dv), g1):
            assert np.array_equal(bits(a[gi]), bits(b))
    uaa.check_device_status()
    # and one group against the oracle
    m = None if mask is None else mask.cpu().numpy().astype(bool)
    qq, kk, vv, dd = (f64(t[1]) for t in (q, k, v, do))
    ro, rl = oracle.attn_fwd(qq, kk, vv, m, scale)
    rdq, rdk, rdv = oracle.attn_bwd(qq, kk, vv, dd, m, scale)
    compare("groups O", f64(o[1]), ro, "o")
    compare("groups LSE", f64(lse[1]), rl, "lse")
    compare("groups dQ", f64(dq[1]), rdq, "dq")
    compare("groups dK", f64(dk[1]), rdk, "dk")
    compare("groups dV", f64(dv[1]), rdv, "dv")


def test_masked_ulysses_exchange_path_end_to_end():
    """The masked Ulysses step through the separate exchanges ("[attention] Add Ulysses
    Anything backward", Validation: the four-rank masked case): every emulated rank holds
    its shard of the key-padding mask; the gathered shards are trimmed and concatenated
    by uaa_assemble_key_mask, and the assembled mask drives the attention of every head
    group (one launch for all groups) in the forward and the backward."""
    lens, cap = (301, 300, 257, 130), 301
    P, B, H, D = 4, 2, 8, 128
    N = sum(lens)
    inp = synth.draw(B, N, H, D, seed=4141)
    g = torch.Generator().manual_seed(4142)
    full_mask = (torch.rand((B, N), generator=g) < 0.7).to(torch.uint8)
    full_mask[1, 301:601] = 0  # rank 1's whole shard masked for batch 1: whole key tiles skipped
    scale = 1.0 / math.sqrt(D)
    mask_sh = oracle.split_key_mask(full_mask.numpy().astype(bool), lens, cap)  # (P, B, cap) per-rank shards
    gathered = torch.from_numpy(mask_sh.astype(np.uint8)).to(DEV)
    key_mask = uaa.assemble_key_mask(gathered, lens)
    assert torch.equal(key_mask.cpu(), full_mask)
    sh = {n: synth.pad_shards(inp[n], lens, cap).to(DEV) for n in ("q", "k", "v", "do")}
    q_sh = sh["q"].requires_grad_(True)
    k_sh = sh["k"].requires_grad_(True)
    v_sh = sh["v"].requires_grad_(True)
    o_sh, lse_g = uaa.ulysses_attention(q_sh, k_sh, v_sh, lens, key_mask, scale)
    o_sh.backward(sh["do"])
    uaa.check_device_status()
    q, k, v, do = (f64(synth.pad_shards(inp[n], lens, cap)) for n in ("q", "k", "v", "do"))
    ro, rl = oracle.ulysses_attn_fwd(q, k, v, lens, cap, mask_sh, scale)
    rdq, rdk, rdv = oracle.ulysses_attn_bwd(q, k, v, do, lens, cap, mask_sh, scale)
    compare("masked ulysses O", f64(o_sh.detach()), ro, "o")
    compare("masked ulysses LSE", f64(lse_g), rl, "lse")
    compare("masked ulysses dQ", f64(q_sh.grad), rdq, "dq")
    compare("masked ulysses dK", f64(k_sh.grad), rdk, "dk")
    compare("masked ulysses dV", f64(v_sh.grad), rdv, "dv")
    offs = np.concatenate([[0], np.cumsum(lens)])
    for p, L in enumerate(lens):
        mp = full_mask.numpy().astype(bool)[:, offs[p]:offs[p] + L]
        for t in (k_sh.grad, v_sh.grad):
            assert (f64(t[p, :, :L])[~mp] == 0).all()
        for t in (o_sh, q_sh.grad, k_sh.grad, v_sh.grad):
            assert (bits(t[p, :, L:]) == 0).all()


def test_autograd_function_marks_lse_non_differentiable():
    inp = synth.draw(1, 64, 2, 64, seed=9)
    q, k, v = (inp[n].to(DEV).requires_grad_(True) for n in ("q", "k", "v"))
    out, lse = uaa.attention(q, k, v)
    assert not lse.requires_grad
    out.backward(inp["do"].to(DEV))
    dq, dk, dv = uaa.attn_bwd(q.detach(), k.detach(), v.detach(), out.detach(), inp["do"].to(DEV), lse)
    assert np.array_equal(bits(k.grad), bits(dk)) and np.array_equal(bits(v.grad), bits(dv))


def test_watchdog_reports_timeout_and_context_survives():
    assert uaa.watchdog_selftest(2000) == 0
    with pytest.raises(uaa.UAAError) as e:
        uaa.check_device_status()
    assert e.value.status == -5
    uaa.check_device_status()  # cleared
    inp = synth.draw(1, 64, 1, 64, seed=1)
    run_gpu(inp, 0.125, None)  # the context is still usable
