"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module holds no attention or re-layout arithmetic: it only draws random
tensors and key-padding lengths, and zero-pads a full sequence into per-rank
shards the way a sequence-parallel caller holds them.

Recipe (the pages' workloads are DiT activations that are not available, so iid
normals stand in for them):

* ``torch.Generator`` (CPU) seeded with ``BASE_SEED + workload index``;
* draw order Q, K, V, dO: each ``torch.randn`` fp32 ``(B, S, H, D)``, rounded
  to bf16 (round-to-nearest-even by torch's conversion);
* then, for masked workloads, one valid-key length per batch,
  ``L_b ~ U{S/2, ..., S}`` (inclusive), giving the prefix mask
  ``mask[b, j] = j < L_b`` (head-broadcast ``(B, 1, 1, S)`` semantics).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BASE_SEED = 20261202


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    B: int
    S: int
    H: int
    D: int
    masked: bool = False
    P: int = 1
    shard_lens: tuple = field(default_factory=tuple)
    cap: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def seed(self) -> int:
        return BASE_SEED + self.index


# The five workloads: a layout trap with H == S, a DiT-like shape with H != S, a
# key-padding-mask case, the Ulysses emulation (4 virtual ranks, uneven final
# shards) and the full DiT-scale layer at N=27280, H=40, D=128.
WORKLOADS = (
    Workload(0, "layout_b2_s16_h16_d64", 2, 16, 16, 64),
    Workload(1, "dit_b2_s1024_h24_d64", 2, 1024, 24, 64),
    Workload(2, "mask_b4_s4096_h24_d128", 4, 4096, 24, 128, masked=True),
    Workload(3, "ulysses_p4_n27280_h40_d128", 1, 27280, 40, 128, P=4,
             shard_lens=(6821, 6821, 6819, 6819), cap=6821),
    Workload(4, "dit_b1_s27280_h40_d128", 1, 27280, 40, 128),
)

EVEN_SHARDS_27280 = (6820, 6820, 6820, 6820)


def workload(name_or_index) -> Workload:
    if isinstance(name_or_index, int):
        return WORKLOADS[name_or_index]
    for w in WORKLOADS:
        if w.name == name_or_index:
            return w
    raise KeyError(name_or_index)


def draw(B, S, H, D, seed, masked=False, with_grad_out=True):
    """Draw bf16 ``q, k, v`` (and ``do``) of shape ``(B, S, H, D)`` plus mask lengths."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    out = {}
    names = ("q", "k", "v", "do") if with_grad_out else ("q", "k", "v")
    for n in names:
        out[n] = torch.randn((B, S, H, D), generator=g, dtype=torch.float32).to(torch.bfloat16)
    if masked:
        lens = torch.randint(S // 2, S + 1, (B,), generator=g)
        out["mask_lens"] = lens
        out["mask"] = (torch.arange(S)[None, :] < lens[:, None]).to(torch.uint8)
    else:
        out["mask_lens"] = None
        out["mask"] = None
    return out


def draw_device(B, S, H, D, seed, device):
    """The same recipe drawn by a seeded generator on ``device`` (for tensors too large to draw
    on the host in reasonable time): bf16 ``q, k, v, do`` of shape ``(B, S, H, D)``, drawn one
    after the other, each as fp32 N(0, 1) rounded to bf16.  A different random stream from
    :func:`draw` for the same seed."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    out = {}
    for n in ("q", "k", "v", "do"):
        out[n] = torch.randn((B, S, H, D), generator=g, dtype=torch.float32, device=device).to(torch.bfloat16)
    return out


def make(w: Workload, with_grad_out=True):
    return draw(w.B, w.S, w.H, w.D, w.seed, w.masked, with_grad_out)


def pad_shards(x, shard_lens, cap):
    """``(B, N, ...)`` -> ``(P, B, cap, ...)``: each rank's contiguous shard, zero-padded."""
    lens = [int(v) for v in shard_lens]
    if sum(lens) != x.shape[1] or max(lens) > cap:
        raise ValueError("bad shard partition")
    out = torch.zeros((len(lens), x.shape[0], cap) + tuple(x.shape[2:]), dtype=x.dtype)
    o = 0
    for p, L in enumerate(lens):
        out[p, :, :L] = x[:, o:o + L]
        o += L
    return out
