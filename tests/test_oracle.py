"""Pins for the fp64 oracle, on the CPU (no GPU, no CUDA extension).

Each check ties the oracle to something other than itself: hand-derived closed
forms (``tests/golden/``), torch's own float64 SDPA and autograd (an independent
library routine), central finite differences, and invariants of softmax
attention and of the Ulysses permutation.  ``test_pins_catch_planted_mistakes``
plants plausible mistakes in a copy of the oracle and checks that the pins fail.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import ref
from ulysses_dit_attention_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# --------------------------------------------------------------------------- golden
def test_golden_two_keys_closed_form():
    doc = json.load(open(os.path.join(GOLDEN, "attention_two_keys.json")))
    for case in doc["cases"]:
        q, k, v, do = (np.array(case[n], dtype=np.float64) for n in ("q", "k", "v", "do"))
        mask = None if case["mask"] is None else np.array(case["mask"], dtype=bool)
        o, lse = oracle.attn_fwd(q, k, v, mask, case["scale"])
        np.testing.assert_allclose(o, case["o"], rtol=0, atol=1e-14, err_msg=case["name"])
        np.testing.assert_allclose(lse, case["lse"], rtol=0, atol=1e-14, err_msg=case["name"])
        dq, dk, dv = oracle.attn_bwd(q, k, v, do, mask, case["scale"])
        for got, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
            np.testing.assert_allclose(got, case[n], rtol=0, atol=1e-14, err_msg=f"{case['name']} {n}")


def test_golden_relayout_index_map():
    doc = json.load(open(os.path.join(GOLDEN, "ulysses_relayout_small.json")))
    x = np.array(doc["x_shards"], dtype=np.float64)
    y = oracle.seq_to_head(x, doc["shard_lens"], doc["cap"])
    np.testing.assert_array_equal(y, np.array(doc["y_groups"], dtype=np.float64))
    back = oracle.head_to_seq(y, doc["shard_lens"], doc["cap"])
    np.testing.assert_array_equal(back, x)
    g = np.array(doc["mask_gathered"], dtype=np.uint8)
    np.testing.assert_array_equal(oracle.assemble_key_mask(g, doc["shard_lens"]), doc["mask_assembled"])
    np.testing.assert_array_equal(oracle.assemble_key_mask_untrimmed(g), doc["mask_untrimmed_defect"])


# --------------------------------------------------------------------------- library routine
def _torch_sdpa(q, k, v, do, mask, scale):
    """torch float64 SDPA (math backend on CPU) + autograd, in BSHD."""
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64).transpose(1, 2).requires_grad_(True) for a in (q, k, v))
    am = None
    if mask is not None:
        am = torch.tensor(mask, dtype=torch.bool)[:, None, None, :]
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=am, scale=scale)
    scores = scale * (tq @ tk.transpose(-1, -2))
    if am is not None:
        scores = scores.masked_fill(~am, float("-inf"))
    lse = torch.logsumexp(scores, dim=-1)
    out.backward(torch.tensor(do, dtype=torch.float64).transpose(1, 2))
    return (out.detach().transpose(1, 2).numpy(), lse.detach().numpy(),
            tq.grad.transpose(1, 2).numpy(), tk.grad.transpose(1, 2).numpy(), tv.grad.transpose(1, 2).numpy())


@pytest.mark.parametrize("B,S,H,D,masked,scale", [
    (2, 16, 16, 8, False, None),      # H == S layout trap shape (scaled down in D)
    (1, 37, 3, 16, True, None),       # ragged length, mask
    (2, 64, 2, 32, True, 0.3),        # explicit non-default scale
])
def test_matches_torch_float64_sdpa(B, S, H, D, masked, scale):
    q, k, v, do = (rnd((B, S, H, D), s) for s in (1, 2, 3, 4))
    mask = None
    if masked:
        lens = np.random.default_rng(5).integers(S // 2, S + 1, size=B)
        mask = np.arange(S)[None, :] < lens[:, None]
    sc = scale if scale is not None else 1.0 / np.sqrt(D)
    o, lse = oracle.attn_fwd(q, k, v, mask, sc, row_block=7)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, mask, sc, row_block=5)
    to, tl, tdq, tdk, tdv = _torch_sdpa(q, k, v, do, mask, sc)
    for a, b in ((o, to), (lse, tl), (dq, tdq), (dk, tdk), (dv, tdv)):
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-11)


# --------------------------------------------------------------------------- finite differences
def _fd_check(mask, seed):
    B, S, H, D = 1, 4, 2, 8
    q, k, v, do = (rnd((B, S, H, D), seed + s) for s in range(4))
    sc = 1.0 / np.sqrt(D)

    def loss(qq, kk, vv):
        o, _ = oracle.attn_fwd(qq, kk, vv, mask, sc)
        return float((o * do).sum())

    dq, dk, dv = oracle.attn_bwd(q, k, v, do, mask, sc)
    h = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            old = x[idx]
            x[idx] = old + h
            lp = loss(q, k, v)
            x[idx] = old - h
            lm = loss(q, k, v)
            x[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        err = np.abs(num - g).max() / max(1.0, np.abs(g).max())
        assert err <= 1e-6, err


def test_finite_differences_unmasked():
    _fd_check(None, 10)


def test_finite_differences_masked():
    _fd_check(np.array([[True, True, False, True]]), 20)


# --------------------------------------------------------------------------- invariants / closed forms
def test_softmax_rows_sum_to_one_and_nonnegative():
    B, S, H, D = 2, 33, 3, 16
    q, k = rnd((B, S, H, D), 1) * 3, rnd((B, S, H, D), 2) * 3
    mask = np.arange(S)[None, :] < np.array([20, 33])[:, None]
    p = oracle.attn_probs(q, k, mask)
    assert (p >= 0).all()
    np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-12)
    assert (p[0, :, :, 20:] == 0).all()


def test_zero_keys_give_column_mean_and_log_length():
    B, S, H, D = 2, 40, 2, 16
    q, v = rnd((B, S, H, D), 1), rnd((B, S, H, D), 2)
    k = np.zeros((B, S, H, D))
    lens = np.array([17, 40])
    mask = np.arange(S)[None, :] < lens[:, None]
    o, lse = oracle.attn_fwd(q, k, v, mask)
    for b in range(B):
        L = lens[b]
        np.testing.assert_allclose(o[b], np.broadcast_to(v[b, :L].mean(0), (S, H, D)), atol=1e-13)
        np.testing.assert_allclose(lse[b], np.log(L), atol=1e-13)


def test_single_valid_key():
    B, S, H, D = 1, 12, 2, 8
    q, k, v, do = (rnd((B, S, H, D), s) for s in range(4))
    mask = np.zeros((B, S), dtype=bool)
    mask[0, 5] = True
    o, lse = oracle.attn_fwd(q, k, v, mask)
    np.testing.assert_allclose(o, np.broadcast_to(v[:, 5:6], o.shape), atol=1e-14)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, mask)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13
    np.testing.assert_allclose(dv[:, 5], do.sum(1), atol=1e-13)
    assert (np.delete(dv, 5, axis=1) == 0).all()


def test_prefix_mask_equals_truncated_keys_and_zero_grads():
    B, S, H, D = 1, 29, 2, 16
    L = 13
    q, k, v, do = (rnd((B, S, H, D), s) for s in range(4))
    mask = np.arange(S)[None, :] < L
    o, lse = oracle.attn_fwd(q, k, v, mask)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, mask)
    # reference: the same queries against only the first L keys
    scale = 1.0 / np.sqrt(D)
    for h in range(H):
        s = scale * q[0, :, h] @ k[0, :L, h].T
        p = np.exp(s - s.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        np.testing.assert_allclose(o[0, :, h], p @ v[0, :L, h], atol=1e-13)
    assert (dk[0, L:] == 0).all() and (dv[0, L:] == 0).all()


def test_dv_is_pt_dout_and_delta_identity():
    B, S, H, D = 2, 24, 3, 8
    q, k, v, do = (rnd((B, S, H, D), s) for s in range(4))
    p = oracle.attn_probs(q, k)
    o, _ = oracle.attn_fwd(q, k, v)
    dq, dk, dv, delta = oracle.attn_bwd(q, k, v, do, return_delta=True)
    for b in range(B):
        for h in range(H):
            np.testing.assert_allclose(dv[b, :, h], p[b, h].T @ do[b, :, h], atol=1e-12)
    # Delta_i = sum_j P_ij dP_ij equals dO_i . O_i
    np.testing.assert_allclose(delta, np.einsum("bshd,bshd->bhs", do, o), atol=1e-12)


def test_fully_masked_row_definition():
    B, S, H, D = 1, 6, 1, 4
    q, k, v, do = (rnd((B, S, H, D), s) for s in range(4))
    mask = np.zeros((B, S), dtype=bool)
    o, lse = oracle.attn_fwd(q, k, v, mask)
    assert (o == 0).all() and np.isneginf(lse).all()
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, mask)
    assert (dq == 0).all() and (dk == 0).all() and (dv == 0).all()


def test_heads_are_independent():
    B, S, H, D = 1, 20, 6, 8
    q, k, v, do = (rnd((B, S, H, D), s) for s in range(4))
    o, lse = oracle.attn_fwd(q, k, v)
    grads = oracle.attn_bwd(q, k, v, do)
    perm = np.array([3, 0, 5, 1, 4, 2])
    o2, lse2 = oracle.attn_fwd(q[:, :, perm], k[:, :, perm], v[:, :, perm])
    np.testing.assert_array_equal(o2, o[:, :, perm])
    np.testing.assert_array_equal(lse2, lse[:, perm])
    sub = [1, 4]
    o3, _ = oracle.attn_fwd(q[:, :, sub], k[:, :, sub], v[:, :, sub])
    np.testing.assert_array_equal(o3, o[:, :, sub])
    g3 = oracle.attn_bwd(q[:, :, sub], k[:, :, sub], v[:, :, sub], do[:, :, sub])
    for a, b in zip(g3, grads):
        np.testing.assert_array_equal(a, b[:, :, sub])


# --------------------------------------------------------------------------- re-layout
@pytest.mark.parametrize("lens,cap", [((6, 6, 6, 6), 6), ((7, 7, 5, 5), 7), ((1, 9, 0, 4), 9)])
def test_relayout_is_a_bijection_and_round_trips(lens, cap):
    P, B, H, D = 4, 2, 8, 3
    N = sum(lens)
    full = np.arange(B * N * H * D, dtype=np.float64).reshape(B, N, H, D) + 1.0
    x = oracle.shard_sequence(full, lens, cap)
    y = oracle.seq_to_head(x, lens, cap)
    assert y.shape == (P, B, N, H // P, D)
    vals = y.ravel()
    assert len(np.unique(vals)) == vals.size == full.size       # every element exactly once
    assert set(vals.tolist()) == set(full.ravel().tolist())
    for g in range(P):                                          # group g = heads of g, all rows
        np.testing.assert_array_equal(y[g], full[:, :, g * (H // P):(g + 1) * (H // P)])
    back = oracle.head_to_seq(y, lens, cap)
    np.testing.assert_array_equal(back, x)
    for p, L in enumerate(lens):
        assert (back[p, :, L:] == 0).all()
    np.testing.assert_array_equal(oracle.unshard_sequence(back, lens), full)


@pytest.mark.parametrize("H,P", [(6, 4), (5, 2), (3, 4)])
def test_relayout_padded_heads(H, P):
    """H % P != 0: heads are zero-padded to P*ceil(H/P) on the way in and dropped on the way back."""
    lens = tuple([4, 3, 4, 2][:P]) if P <= 4 else None
    cap = max(lens)
    B, D = 2, 3
    N = sum(lens)
    hg = -(-H // P)
    full = np.arange(B * N * H * D, dtype=np.float64).reshape(B, N, H, D) + 1.0
    x = oracle.shard_sequence(full, lens, cap)
    y = oracle.seq_to_head(x, lens, cap)
    assert y.shape == (P, B, N, hg, D)
    for g in range(P):
        for hh in range(hg):
            h = g * hg + hh
            if h < H:
                np.testing.assert_array_equal(y[g, :, :, hh], full[:, :, h])
            else:
                assert (y[g, :, :, hh] == 0).all()      # padding head
    nz = y[y != 0]
    assert nz.size == full.size and len(np.unique(nz)) == full.size  # each real element exactly once
    back = oracle.head_to_seq(y, lens, cap, H)
    assert back.shape == x.shape
    np.testing.assert_array_equal(back, x)


def test_ulysses_composition_with_padded_heads():
    lens, cap = (5, 4, 4, 3), 5
    B, N, H, D = 1, 16, 6, 8
    q, k, v, do = (rnd((B, N, H, D), s + 10) for s in range(4))
    sh = [oracle.shard_sequence(t, lens, cap) for t in (q, k, v, do)]
    o_sh, lse_g = oracle.ulysses_attn_fwd(sh[0], sh[1], sh[2], lens, cap)
    o, lse = oracle.attn_fwd(q, k, v)
    np.testing.assert_allclose(oracle.unshard_sequence(o_sh, lens), o, atol=1e-14)
    assert lse_g.shape == (4, B, 2, N)
    for h in range(H):
        np.testing.assert_allclose(lse_g[h // 2][:, h % 2], lse[:, h], atol=1e-14)
    np.testing.assert_allclose(lse_g[3], np.log(N), atol=1e-14)  # zero heads: uniform over all keys
    dq_sh, dk_sh, dv_sh = oracle.ulysses_attn_bwd(*sh, lens, cap)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do)
    for a, b in ((dq_sh, dq), (dk_sh, dk), (dv_sh, dv)):
        np.testing.assert_allclose(oracle.unshard_sequence(a, lens), b, atol=1e-13)


def test_relayout_matches_synth_padding():
    lens, cap = (5, 5, 4, 3), 5
    full = torch.arange(2 * 17 * 4 * 2, dtype=torch.float32).reshape(2, 17, 4, 2)
    a = synth.pad_shards(full, lens, cap).numpy().astype(np.float64)
    b = oracle.shard_sequence(full.numpy().astype(np.float64), lens, cap)
    np.testing.assert_array_equal(a, b)


def test_mask_assembly_trim_before_concat():
    lens, cap = (6821, 6821, 6819, 6819), 6821
    rng = np.random.default_rng(7)
    mask = (rng.random((1, sum(lens))) < 0.7).astype(np.uint8)
    g = oracle.split_key_mask(mask, lens, cap)
    assert g.shape == (4, 1, cap)
    np.testing.assert_array_equal(oracle.assemble_key_mask(g, lens), mask)
    bad = oracle.assemble_key_mask_untrimmed(g)
    assert bad.shape != mask.shape  # regression sentinel: the untrimmed concat is wrong


def test_ulysses_composition_equals_full_attention():
    lens, cap = (5, 5, 3, 3), 5
    B, N, H, D = 1, 16, 8, 8
    q, k, v, do = (rnd((B, N, H, D), s) for s in range(4))
    mask = (np.arange(N) < 12)[None, :]
    sh = [oracle.shard_sequence(t, lens, cap) for t in (q, k, v, do)]
    msh = oracle.split_key_mask(mask.astype(np.uint8), lens, cap)
    o_sh, lse_g = oracle.ulysses_attn_fwd(sh[0], sh[1], sh[2], lens, cap, msh)
    o, lse = oracle.attn_fwd(q, k, v, mask)
    np.testing.assert_allclose(oracle.unshard_sequence(o_sh, lens), o, atol=1e-14)
    for g in range(4):
        np.testing.assert_allclose(lse_g[g], lse[:, 2 * g:2 * g + 2], atol=1e-14)
    dq_sh, dk_sh, dv_sh = oracle.ulysses_attn_bwd(*sh, lens, cap, msh)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, mask)
    for a, b in ((dq_sh, dq), (dk_sh, dk), (dv_sh, dv)):
        np.testing.assert_allclose(oracle.unshard_sequence(a, lens), b, atol=1e-13)


def test_key_bias_rejects_per_head_mask():
    with pytest.raises(ValueError):
        ref.key_bias(np.ones((2, 3, 1, 5), dtype=bool), 2, 5)
    bias = ref.key_bias(np.ones((2, 1, 1, 5), dtype=bool), 2, 5)
    assert (bias == 0).all()


# --------------------------------------------------------------------------- planted mistakes
def _mutant_bwd(kind):
    def bwd(q, k, v, do, key_mask=None, scale=None, row_block=1024, return_delta=False):
        B, S, H, D = q.shape
        scale = 1.0 / np.sqrt(D) if scale is None else scale
        bias = ref.key_bias(key_mask, B, S)
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        for b in range(B):
            for h in range(H):
                qb, kh, vh, dob = q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h]
                s = scale * qb @ kh.T + bias[b][None, :]
                p = np.exp(s - s.max(1, keepdims=True))
                p /= p.sum(1, keepdims=True)
                dp = dob @ vh.T
                d_i = (p * dp).sum(1)
                if kind == "drop_delta":
                    d_i = 0 * d_i
                ds = p * (dp - d_i[:, None])
                dv[b, :, h] = (p if kind == "p_not_transposed" else p.T) @ dob
                dq[b, :, h] = (1.0 if kind == "no_scale_dq" else scale) * ds @ kh
                dk[b, :, h] = scale * ds.T @ (kh if kind == "k_for_q" else qb)
        return dq, dk, dv
    return bwd


def _mutant_fwd(kind):
    def fwd(q, k, v, key_mask=None, scale=None, row_block=1024):
        B, S, H, D = q.shape
        scale = 1.0 / np.sqrt(D) if scale is None else scale
        bias = ref.key_bias(key_mask, B, S)
        if kind == "mask_inverted":
            bias = np.where(np.isinf(bias), 0.0, -np.inf)
        o = np.zeros_like(q)
        lse = np.zeros((B, H, S))
        for b in range(B):
            for h in range(H):
                s = (1.0 if kind == "no_scale" else scale) * q[b, :, h] @ k[b, :, h].T + bias[b][None, :]
                m = s.max(1, keepdims=True)
                e = np.exp(s - m)
                p = e / e.sum(1, keepdims=True)
                o[b, :, h] = p @ v[b, :, h]
                lse[b, h] = (m[:, 0] + np.log(e.sum(1))) * (np.log2(np.e) if kind == "lse_base2" else 1.0)
        return o, lse
    return fwd


@pytest.mark.parametrize("kind", ["drop_delta", "p_not_transposed", "no_scale_dq", "k_for_q"])
def test_pins_catch_planted_backward_mistakes(kind, monkeypatch):
    monkeypatch.setattr(oracle, "attn_bwd", _mutant_bwd(kind))
    failed = False
    try:
        _fd_check(None, 10)
        test_golden_two_keys_closed_form()
    except AssertionError:
        failed = True
    assert failed, kind


@pytest.mark.parametrize("kind", ["no_scale", "mask_inverted", "lse_base2"])
def test_pins_catch_planted_forward_mistakes(kind, monkeypatch):
    monkeypatch.setattr(oracle, "attn_fwd", _mutant_fwd(kind))
    failed = False
    try:
        with np.errstate(all="ignore"):
            test_golden_two_keys_closed_form()
            test_zero_keys_give_column_mean_and_log_length()
    except AssertionError:
        failed = True
    assert failed, kind


# --------------------------------------------------------------------------- inputs
def test_synth_is_seeded_and_bf16():
    w = synth.workload(0)
    a, b = synth.make(w), synth.make(w)
    for n in ("q", "k", "v", "do"):
        assert a[n].dtype == torch.bfloat16 and a[n].shape == (2, 16, 16, 64)
        assert torch.equal(a[n], b[n])
    m = synth.make(synth.workload(2), with_grad_out=False)
    lens = m["mask_lens"]
    assert ((lens >= 2048) & (lens <= 4096)).all()
    assert m["mask"].shape == (4, 4096)
    assert torch.equal(m["mask"].sum(1).to(torch.int64), lens.to(torch.int64))


def test_query_row_subset_is_exact():
    B, S, H, D = 1, 50, 2, 8
    q, k, v, do = (rnd((B, S, H, D), s) for s in range(4))
    mask = (np.arange(S) < 41)[None, :]
    o, lse = oracle.attn_fwd(q, k, v, mask)
    dq, _, _ = oracle.attn_bwd(q, k, v, do, mask)
    rows = np.array([0, 7, 33, 49])
    o2, lse2 = oracle.attn_fwd(q[:, rows], k, v, mask)
    dq2, _, _ = oracle.attn_bwd(q[:, rows], k, v, do[:, rows], mask)
    np.testing.assert_array_equal(o2, o[:, rows])
    np.testing.assert_array_equal(lse2, lse[:, :, rows])
    np.testing.assert_allclose(dq2, dq[:, rows], atol=1e-15)
