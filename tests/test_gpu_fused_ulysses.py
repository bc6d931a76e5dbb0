"""Ulysses attention with the exchanges fused into the attention kernels, on the
GPU through the C ABI, against the fp64 oracle's own Ulysses composition
(seq->head exchange, attention per head group, head->seq exchange).

The fused kernels read 128-row tiles straight from the sequence shards (a tile
never straddles two shards, so the last tile of each shard is partial) and
write O, dQ, dK, dV back into the shards.  The cases cover partial tiles in
every shard, empty shards (leading, inner, last), a shard of one row, shards
ending exactly on a tile boundary, P = 1 and the maximum P = 8, key masks, and
the full-size uneven-shard Ulysses workload on sampled heads.
"""
import numpy as np
import pytest
import torch

import oracle
import ulysses_dit_attention_gb300 as uaa
from ulysses_dit_attention_gb300 import synth
from helpers import bits, compare, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def lse_full(lse_groups, H):
    """Oracle LSE, head-sharded (P, B, Hg, N) -> (B, H, N)."""
    P, B, Hg, N = lse_groups.shape
    out = np.empty((B, H, N))
    for g in range(P):
        for hh in range(Hg):
            if g * Hg + hh < H:
                out[:, g * Hg + hh] = lse_groups[g, :, hh]
    return out


CASES = [
    # P, shard_lens, cap, B, H, D, mask kind
    (4, [70, 70, 67, 66], 70, 2, 8, 128, None),          # every shard one partial tile
    (4, [130, 129, 0, 200], 200, 1, 4, 64, "random"),    # an empty shard, two-tile shards, random mask
    (3, [257, 1, 128], 300, 2, 3, 128, "random"),        # a one-row shard, a shard ending on a tile boundary
    (1, [300], 320, 1, 2, 64, None),                     # one shard with padding rows
    (8, [50, 50, 50, 50, 50, 50, 50, 33], 64, 1, 8, 128, None),  # the largest P
    (2, [129, 127], 130, 2, 2, 128, "prefix"),           # prefix key mask over the sequence
    (2, [100, 0], 100, 1, 2, 128, None),                 # empty last shard: the pair's second query tile is past the end
    (3, [0, 0, 70], 70, 2, 2, 64, "random"),             # empty leading shards
    (2, [128, 256], 256, 1, 3, 128, None),               # every shard a whole number of tiles
    (3, [200, 300, 140], 300, 2, 2, 128, "holes"),       # whole key tiles masked inside shards 1 and 2
    (3, [200, 300, 140], 300, 1, 2, 64, "holes"),
]


@pytest.mark.parametrize("P,lens,cap,B,H,D,kind", CASES)
def test_fused_ulysses_matches_the_oracle(P, lens, cap, B, H, D, kind):
    N = sum(lens)
    scale = 1.0 / np.sqrt(D)
    inp = synth.draw(B, N, H, D, seed=7000 + P * 31 + N)
    sh = {n: synth.pad_shards(inp[n], lens, cap) for n in ("q", "k", "v", "do")}
    mask = None
    if kind == "random":
        g = torch.Generator().manual_seed(N)
        mask = (torch.rand((B, N), generator=g) < 0.7).to(torch.uint8)
    elif kind == "prefix":
        mask = (torch.arange(N)[None, :] < torch.tensor([N // 2 + 3, N])[:B, None]).to(torch.uint8)
    elif kind == "holes":
        # the first tile of shard 1 (positions 200..327) and of shard 2 (500..627) hold no
        # attended key, between partly attended tiles
        g = torch.Generator().manual_seed(N + 1)
        mask = (torch.rand((B, N), generator=g) < 0.7).to(torch.uint8)
        mask[:, 200:328] = 0
        mask[:, 500:628] = 0
    dsh = {n: t.to(DEV) for n, t in sh.items()}
    dmask = None if mask is None else mask.to(DEV)
    o_sh, lse = uaa.ulysses_attn_fwd(dsh["q"], dsh["k"], dsh["v"], lens, dmask, scale)
    dq, dk, dv = uaa.ulysses_attn_bwd(dsh["q"], dsh["k"], dsh["v"], o_sh, dsh["do"], lse, lens, dmask, scale)
    uaa.check_device_status()

    q, k, v, do = (f64(sh[n]) for n in ("q", "k", "v", "do"))
    mask_sh = None if mask is None else oracle.split_key_mask(mask.numpy().astype(bool), lens, cap)
    ro, rl = oracle.ulysses_attn_fwd(q, k, v, lens, cap, mask_sh, scale)
    rdq, rdk, rdv = oracle.ulysses_attn_bwd(q, k, v, do, lens, cap, mask_sh, scale)
    label = f"P={P} lens={lens}"
    compare(f"{label} O", f64(o_sh), ro, "o")
    compare(f"{label} LSE", f64(lse), lse_full(rl, H), "lse")
    compare(f"{label} dQ", f64(dq), rdq, "dq")
    compare(f"{label} dK", f64(dk), rdk, "dk")
    compare(f"{label} dV", f64(dv), rdv, "dv")
    # padding rows are exactly zero; masked keys get exactly zero dK / dV
    for p, L in enumerate(lens):
        for t in (o_sh, dq, dk, dv):
            assert (bits(t[p, :, L:]) == 0).all()
    if mask is not None:
        m = mask.numpy().astype(bool)
        offs = np.concatenate([[0], np.cumsum(lens)])
        for p, L in enumerate(lens):
            mp = m[:, offs[p]:offs[p] + L]
            for t in (dk, dv):
                tp = f64(t[p, :, :L])
                assert (tp[~mp] == 0).all()


def test_fused_ulysses_is_deterministic():
    lens, cap, B, H, D = [300, 170, 299], 300, 1, 4, 128
    inp = synth.draw(B, sum(lens), H, D, seed=91)
    sh = {n: synth.pad_shards(inp[n], lens, cap).to(DEV) for n in ("q", "k", "v", "do")}
    runs = []
    for _ in range(2):
        o, lse = uaa.ulysses_attn_fwd(sh["q"], sh["k"], sh["v"], lens)
        grads = uaa.ulysses_attn_bwd(sh["q"], sh["k"], sh["v"], o, sh["do"], lse, lens)
        runs.append([bits(t) for t in (o, lse) + grads])
    uaa.check_device_status()
    for a, b in zip(*runs):
        assert np.array_equal(a, b)


def test_fused_ulysses_workload_sampled_heads():
    """The uneven-shard Ulysses workload (N = 27280 as 6821, 6821, 6819, 6819; H = 40,
    D = 128) through the fused autograd path; heads are independent, so the oracle
    evaluates two of them on the unsharded sequence."""
    w = synth.workload("ulysses_p4_n27280_h40_d128")
    inp = synth.make(w)
    lens, cap = w.shard_lens, w.cap
    sh = {n: synth.pad_shards(inp[n], lens, cap).to(DEV) for n in ("q", "k", "v", "do")}
    q_sh = sh["q"].requires_grad_(True)
    k_sh = sh["k"].requires_grad_(True)
    v_sh = sh["v"].requires_grad_(True)
    o_sh, lse = uaa.ulysses_attention_fused(q_sh, k_sh, v_sh, lens, None, w.scale)
    o_sh.backward(sh["do"])
    uaa.check_device_status()
    for p, L in enumerate(lens):
        for t in (o_sh, q_sh.grad, k_sh.grad, v_sh.grad):
            assert (bits(t[p, :, L:]) == 0).all()

    def unshard(t):
        return torch.cat([t[p, :, :L] for p, L in enumerate(lens)], dim=1)

    heads = [1, w.H - 3]
    q, k, v, do = (f64(inp[n])[:, :, heads] for n in ("q", "k", "v", "do"))
    ro, rl = oracle.attn_fwd(q, k, v, None, w.scale)
    rdq, rdk, rdv = oracle.attn_bwd(q, k, v, do, None, w.scale)
    compare("fused ulysses O", f64(unshard(o_sh.detach()))[:, :, heads], ro, "o")
    compare("fused ulysses LSE", f64(lse)[:, heads], rl, "lse")
    compare("fused ulysses dQ", f64(unshard(q_sh.grad))[:, :, heads], rdq, "dq")
    compare("fused ulysses dK", f64(unshard(k_sh.grad))[:, :, heads], rdk, "dk")
    compare("fused ulysses dV", f64(unshard(v_sh.grad))[:, :, heads], rdv, "dv")
