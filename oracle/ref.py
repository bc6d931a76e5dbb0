"""Plain fp64 CPU oracle for the Ulysses DiT attention hot path.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py`` (its ``cpu_baseline`` leg and its ``--impl reference`` arm) may
import or run anything in this package.  It shares no code with the CUDA path
(``ulysses_dit_attention_gb300``) and imports nothing from it: it uses NumPy
only and works on float64 arrays.  Callers convert the same bf16 values the GPU
consumes to float64 (exact) before calling in.

Every function states the passage of the source pages it follows.  The pages are
three pull-request discussions:

* "[attention] Add Ulysses Anything backward" (diffusers PR 14834), cited "UAA-bwd";
* "Add fast-ulysses attention backend" (LightX2V PR 1234), cited "fast-ulysses";
* "Fix double transpose of K/V in templated attention backward" (diffusers
  PR 14341), cited "double-transpose".

The method (tiled online-softmax attention, Ulysses sharding) reaches exactly
the plain result of softmax attention, so this oracle is that plain definition
written out: dense scores per query-row block, a max-subtracted softmax, and
the textbook softmax-attention gradient.  No tiling over keys, no online
rescaling, no fusion.

Parity pins: every function here is pinned by ``tests/test_oracle.py``
(closed forms, a hand-derived worked example under ``tests/golden/``, torch's
own float64 SDPA + autograd, central finite differences, invariants).  No
function is "parity unpinned".

Conventions (readings of what the pages leave open):
* tensors are BSHD ``(B, S, H, D)`` -- the forward op returns its output in
  BSHD ("double-transpose", description paragraph on the forward/backward op
  contract);
* ``lse`` is ``(B, H, S)``, the natural log of the sum of exponentials of the
  *scaled* scores (bias included);
* ``key_mask`` is ``(B, S)`` of bools/0-1, True = attend, shared by all heads --
  the head-broadcast ``(B, 1, 1, S)`` mask ("UAA-bwd", Unsupported cases,
  per-head masks paragraph); it becomes an additive 0 / -inf bias
  ("double-transpose", follow-up item 2, bool mask to additive bias);
* a query row whose keys are all masked has O = 0, LSE = -inf and contributes
  no gradient (the pages never reach this case);
* ``attn_fwd`` / ``attn_bwd`` accept a query block of ``Sq`` rows against
  ``Sk`` keys (rows are independent, so the tests can evaluate sampled query
  rows of a long sequence exactly; ``dK``/``dV`` are then the contribution of
  those rows only).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "key_bias",
    "attn_fwd",
    "attn_bwd",
    "attn_probs",
    "shard_sequence",
    "unshard_sequence",
    "seq_to_head",
    "head_to_seq",
    "split_key_mask",
    "assemble_key_mask",
    "assemble_key_mask_untrimmed",
    "ulysses_attn_fwd",
    "ulysses_attn_bwd",
]

_ROW_BLOCK = 1024


def _check_bshd(*xs):
    for x in xs:
        if x.ndim != 4:
            raise ValueError(f"expected a (B, S, H, D) array, got shape {x.shape}")
        if x.dtype != np.float64:
            raise TypeError("the oracle works in float64; convert the bf16 inputs first")


def key_bias(key_mask, B, S):
    """Additive key bias ``(B, S)``: 0 where the mask is True, -inf where False.

    "double-transpose", follow-up item 2: a bool attention mask has to become an
    additive -inf/0 bias before it enters the attention kernel.  ``None`` means
    every key is attended.
    """
    if key_mask is None:
        return np.zeros((B, S), dtype=np.float64)
    m = np.asarray(key_mask)
    if m.ndim == 4:
        # (B, 1, 1, S) head-broadcast form; a per-head (B, H>1, 1, S) mask cannot
        # be sharded across heads ("UAA-bwd", Unsupported cases, per-head masks).
        if m.shape[1] != 1 or m.shape[2] != 1:
            raise ValueError("only head-broadcast (B, 1, 1, S) key masks are supported")
        m = m[:, 0, 0, :]
    if m.shape != (B, S):
        raise ValueError(f"key mask shape {m.shape} does not match (B, S) = {(B, S)}")
    return np.where(m.astype(bool), 0.0, -np.inf)


def _scores(qb, kh, bias_b, scale):
    # s_ij = scale * q_i . k_j + bias_j  (plain definition of SDPA scores)
    return scale * (qb @ kh.T) + bias_b[None, :]


def _row_lse(s):
    """Natural log-sum-exp of each row of ``s``; -inf for an all -inf row."""
    m = s.max(axis=1)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    tot = np.exp(s - m_safe[:, None]).sum(axis=1)
    with np.errstate(divide="ignore"):
        lse = m_safe + np.log(tot)
    return np.where(finite, lse, -np.inf)


def _probs_from_lse(s, lse):
    # P_ij = exp(s_ij - LSE_i); rows with LSE = -inf (all keys masked) are all zero.
    finite = np.isfinite(lse)
    lse_safe = np.where(finite, lse, 0.0)
    p = np.exp(s - lse_safe[:, None])
    p[~finite, :] = 0.0
    return p


def attn_fwd(q, k, v, key_mask=None, scale=None, row_block=_ROW_BLOCK):
    """Non-causal multi-head SDPA forward in BSHD; returns ``(O, LSE)``.

    "double-transpose", description: the forward op returns ``out`` in BSHD;
    follow-up item 1: the forward must also produce the log-sum-exp, which the
    backward consumes ("UAA-bwd", What does this PR do: the auxiliary LSE output
    is non-differentiable).  Definition, per (b, h):
    ``s_ij = scale * q_i . k_j + bias_j``, ``LSE_i = ln sum_j exp(s_ij)``,
    ``P_ij = exp(s_ij - LSE_i)``, ``O_i = sum_j P_ij v_j``.
    """
    _check_bshd(q, k, v)
    B, S, H, D = q.shape
    Sk = k.shape[1]
    if k.shape != (B, Sk, H, D) or v.shape != (B, Sk, H, D):
        raise ValueError("k and v must be (B, Sk, H, D) with q's B, H, D")
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    bias = key_bias(key_mask, B, Sk)
    o = np.zeros((B, S, H, D), dtype=np.float64)
    lse = np.zeros((B, H, S), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            kh = k[b, :, h, :]
            vh = v[b, :, h, :]
            for i0 in range(0, S, row_block):
                i1 = min(S, i0 + row_block)
                s = _scores(q[b, i0:i1, h, :], kh, bias[b], scale)
                l_i = _row_lse(s)
                p = _probs_from_lse(s, l_i)
                o[b, i0:i1, h, :] = p @ vh
                lse[b, h, i0:i1] = l_i
    return o, lse


def attn_probs(q, k, key_mask=None, scale=None):
    """Dense softmax matrix ``P`` of shape ``(B, H, S, S)`` (small inputs only)."""
    _check_bshd(q, k)
    B, S, H, D = q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    bias = key_bias(key_mask, B, S)
    p = np.zeros((B, H, S, S), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            s = _scores(q[b, :, h, :], k[b, :, h, :], bias[b], scale)
            p[b, h] = _probs_from_lse(s, _row_lse(s))
    return p


def attn_bwd(q, k, v, do, key_mask=None, scale=None, row_block=_ROW_BLOCK, return_delta=False):
    """Textbook softmax-attention gradient; returns ``(dQ, dK, dV)``.

    "double-transpose", description: the backward op takes the saved Q/K/V
    (all in one layout), the output gradient and the LSE, and returns dQ/dK/dV
    ("Test" paragraph: checked against an eager reference).  Per (b, h):
    ``dV_j = sum_i P_ij dO_i``; ``dP_ij = dO_i . v_j``;
    ``Delta_i = sum_j P_ij dP_ij``; ``dS_ij = P_ij (dP_ij - Delta_i)``;
    ``dQ_i = scale sum_j dS_ij k_j``; ``dK_j = scale sum_i dS_ij q_i``.

    ``Delta`` is formed from this function's own ``P`` and ``dP`` (not from the
    shortcut ``rowsum(dO * O)``), so that the identity between the two stays a
    separate check.  With ``return_delta`` the ``(B, H, S)`` Delta is returned too.
    """
    _check_bshd(q, k, v, do)
    B, S, H, D = q.shape
    Sk = k.shape[1]
    if k.shape != (B, Sk, H, D) or v.shape != (B, Sk, H, D) or do.shape != q.shape:
        raise ValueError("k, v must be (B, Sk, H, D) and do must match q")
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    bias = key_bias(key_mask, B, Sk)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    delta = np.zeros((B, H, S), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            kh = k[b, :, h, :]
            vh = v[b, :, h, :]
            for i0 in range(0, S, row_block):
                i1 = min(S, i0 + row_block)
                qb = q[b, i0:i1, h, :]
                dob = do[b, i0:i1, h, :]
                s = _scores(qb, kh, bias[b], scale)
                p = _probs_from_lse(s, _row_lse(s))
                dv[b, :, h, :] += p.T @ dob
                dp = dob @ vh.T
                d_i = (p * dp).sum(axis=1)
                ds = p * (dp - d_i[:, None])
                dq[b, i0:i1, h, :] = scale * (ds @ kh)
                dk[b, :, h, :] += scale * (ds.T @ qb)
                delta[b, h, i0:i1] = d_i
    if return_delta:
        return dq, dk, dv, delta
    return dq, dk, dv


# ---------------------------------------------------------------------------
# Ulysses re-layout ("UAA-bwd", What does this PR do; "fast-ulysses", Summary).
#
# P ranks each hold a contiguous sequence shard of length L_p (uneven lengths
# allowed: "Ulysses Anything"), padded to a common capacity ``cap`` for the
# all-to-all transport.  The forward exchange turns the seq-sharded
# (B, L_p, H, D) shards into head-sharded (B, N, H/P, D) groups with
# N = sum_p L_p; group g owns heads [g*H/P, (g+1)*H/P).  The inverse exchange
# restores outputs/gradients to the seq-sharded form and pads them again.
# On one device the exchange is a pure index permutation.
# ---------------------------------------------------------------------------


def _offsets(shard_lens):
    lens = [int(x) for x in shard_lens]
    if any(L < 0 for L in lens):
        raise ValueError("shard lengths must be non-negative")
    offs = [0]
    for L in lens:
        offs.append(offs[-1] + L)
    return lens, offs


def shard_sequence(x, shard_lens, cap):
    """Split a full ``(B, N, ...)`` sequence into ``(P, B, cap, ...)`` zero-padded shards."""
    lens, offs = _offsets(shard_lens)
    if offs[-1] != x.shape[1]:
        raise ValueError("shard lengths must sum to the sequence length")
    if max(lens) > cap:
        raise ValueError("a shard is longer than the capacity")
    out = np.zeros((len(lens), x.shape[0], cap) + x.shape[2:], dtype=x.dtype)
    for p, L in enumerate(lens):
        out[p, :, :L] = x[:, offs[p]:offs[p] + L]
    return out


def unshard_sequence(shards, shard_lens):
    """Concatenate the valid rows of ``(P, B, cap, ...)`` shards into ``(B, N, ...)``."""
    lens, _ = _offsets(shard_lens)
    return np.concatenate([shards[p, :, :L] for p, L in enumerate(lens)], axis=1)


def seq_to_head(x, shard_lens, cap):
    """Forward Ulysses exchange: ``(P, B, cap, H, D)`` shards -> ``(P, B, N, Hg, D)`` groups.

    ``Hg = ceil(H / P)``.  ``y[g, b, off_p + s, h', :] = x[p, b, s, g*Hg + h', :]``
    for ``s < L_p`` and ``g*Hg + h' < H``; heads ``g*Hg + h' >= H`` are zero:
    every rank sends head group g of its shard to rank g, which concatenates the
    shards it receives in rank order, trimmed to their true lengths ("UAA-bwd",
    What does this PR do: reuse of the all-to-all helpers with the saved
    partition metadata; the head dimension is padded with zero heads to a
    multiple of P when P does not divide H -- the padded-head layouts of Ulysses
    Anything, "UAA-bwd", What does this PR do and Tests).
    """
    P, B, C, H, D = x.shape
    lens, _ = _offsets(shard_lens)
    if len(lens) != P or C != cap:
        raise ValueError("shard buffer does not match shard_lens / cap")
    hg = -(-H // P)
    if hg * P != H:
        pad = np.zeros((P, B, C, hg * P - H, D), dtype=x.dtype)
        x = np.concatenate([x, pad], axis=3)
    groups = []
    for g in range(P):
        parts = [x[p, :, :lens[p], g * hg:(g + 1) * hg, :] for p in range(P)]
        groups.append(np.concatenate(parts, axis=1))
    return np.stack(groups, axis=0)


def head_to_seq(y, shard_lens, cap, H=None):
    """Inverse Ulysses exchange: ``(P, B, N, Hg, D)`` groups -> ``(P, B, cap, H, D)`` shards.

    Rows ``s >= L_p`` of shard p (transport padding) are zero; the zero padding
    heads (``H < P*Hg``) are dropped.  ``H`` defaults to ``P*Hg``.  "UAA-bwd",
    What does this PR do: the outputs and the Q/K/V gradients are restored to
    the sequence-sharded layout by the inverse all-to-all.
    """
    P, B, N, hg, D = y.shape
    lens, offs = _offsets(shard_lens)
    if len(lens) != P or offs[-1] != N:
        raise ValueError("group buffer does not match shard_lens")
    if max(lens) > cap:
        raise ValueError("a shard is longer than the capacity")
    H = P * hg if H is None else int(H)
    if not ((hg - 1) * P < H <= P * hg):
        raise ValueError("H does not match the group size")
    x = np.zeros((P, B, cap, P * hg, D), dtype=y.dtype)
    for p in range(P):
        for g in range(P):
            x[p, :, :lens[p], g * hg:(g + 1) * hg, :] = y[g, :, offs[p]:offs[p] + lens[p]]
    return x[:, :, :, :H]


def split_key_mask(mask, shard_lens, cap):
    """Key mask ``(B, N)`` -> per-rank padded mask shards ``(P, B, cap)`` (padding = 0)."""
    m = np.asarray(mask)
    return shard_sequence(m[:, :, None], shard_lens, cap)[..., 0]


def assemble_key_mask(gathered, shard_lens):
    """Global key mask from gathered padded shards, trimming each shard first.

    "UAA-bwd", What does this PR do: uneven local key-padding mask assembly is
    fixed by trimming every gathered shard to its true length before the
    concatenation (Validation: the four-rank masked case exposed the defect).
    ``gathered`` is ``(P, B, cap)``; the result is ``(B, N)``.
    """
    lens, _ = _offsets(shard_lens)
    if gathered.shape[0] != len(lens):
        raise ValueError("gathered mask does not match shard_lens")
    return np.concatenate([gathered[p, :, :L] for p, L in enumerate(lens)], axis=1)


def assemble_key_mask_untrimmed(gathered):
    """The defective assembly the pages fix: concatenate padded shards as-is.

    Kept only as a regression sentinel: with uneven shards it gives a mask of the
    wrong length whose entries after the first padded shard are shifted.
    """
    return np.concatenate(list(gathered), axis=1)


def ulysses_attn_fwd(q_sh, k_sh, v_sh, shard_lens, cap, mask_sh=None, scale=None):
    """Ulysses attention forward on P emulated ranks.

    seq->head exchange of Q/K/V, attention per head group (the mask, gathered
    from its shards and trimmed, is shared by all heads), head->seq exchange
    of O.  LSE is returned head-sharded ``(P, B, Hg, N)``, as each rank keeps
    it (rows of padding heads included).  "UAA-bwd", What does this PR do.
    """
    H = q_sh.shape[3]
    yq = seq_to_head(q_sh, shard_lens, cap)
    yk = seq_to_head(k_sh, shard_lens, cap)
    yv = seq_to_head(v_sh, shard_lens, cap)
    mask = None if mask_sh is None else assemble_key_mask(mask_sh, shard_lens)
    P = yq.shape[0]
    outs, lses = [], []
    for g in range(P):
        o, lse = attn_fwd(yq[g], yk[g], yv[g], mask, scale)
        outs.append(o)
        lses.append(lse)
    return head_to_seq(np.stack(outs), shard_lens, cap, H), np.stack(lses)


def ulysses_attn_bwd(q_sh, k_sh, v_sh, do_sh, shard_lens, cap, mask_sh=None, scale=None):
    """Ulysses attention backward on P emulated ranks.

    seq->head exchange of dO, attention backward per head group, head->seq
    exchange of dQ (query partition) and dK/dV (key partition; self-attention
    here, so both partitions are ``shard_lens``).  "UAA-bwd", What does this
    PR do.
    """
    H = q_sh.shape[3]
    yq = seq_to_head(q_sh, shard_lens, cap)
    yk = seq_to_head(k_sh, shard_lens, cap)
    yv = seq_to_head(v_sh, shard_lens, cap)
    ydo = seq_to_head(do_sh, shard_lens, cap)
    mask = None if mask_sh is None else assemble_key_mask(mask_sh, shard_lens)
    P = yq.shape[0]
    dqs, dks, dvs = [], [], []
    for g in range(P):
        dq, dk, dv = attn_bwd(yq[g], yk[g], yv[g], ydo[g], mask, scale)
        dqs.append(dq)
        dks.append(dk)
        dvs.append(dv)
    return (head_to_seq(np.stack(dqs), shard_lens, cap, H),
            head_to_seq(np.stack(dks), shard_lens, cap, H),
            head_to_seq(np.stack(dvs), shard_lens, cap, H))
