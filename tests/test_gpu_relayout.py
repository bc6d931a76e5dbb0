"""GPU re-layout and mask-assembly kernels vs the oracle, bit for bit.

Covers even and uneven (Ulysses Anything) partitions, an empty shard, P = 1,
D = 64/128, fp32 elements, the zeroed transport padding, padded heads
(P does not divide H), and the full N = 27280, H = 40, D = 128 workload with
shards (6821, 6821, 6819, 6819).
"""
import numpy as np
import pytest
import torch

import oracle
import ulysses_dit_attention_gb300 as uaa
from ulysses_dit_attention_gb300 import synth
from helpers import bits

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _shards(B, lens, cap, H, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    full = torch.randn((B, sum(lens), H, D), generator=g).to(dtype)
    return full, synth.pad_shards(full, lens, cap)


CASES = [
    # (B, lens, cap, H, D, dtype)
    (1, (6821, 6821, 6819, 6819), 6821, 40, 128, torch.bfloat16),
    (1, (6820, 6820, 6820, 6820), 6820, 40, 128, torch.bfloat16),
    (2, (7, 7, 5, 5), 8, 8, 64, torch.bfloat16),
    (1, (1, 9, 0, 4), 9, 4, 128, torch.bfloat16),
    (3, (33,), 40, 6, 64, torch.bfloat16),
    (2, (5, 3), 5, 4, 64, torch.float32),
    # padded heads: P does not divide H
    (2, (7, 7, 5, 5), 8, 6, 64, torch.bfloat16),
    (1, (5, 3, 4), 5, 8, 128, torch.bfloat16),
    (1, (6821, 6821, 6819, 6819), 6821, 42, 128, torch.bfloat16),
]


@pytest.mark.parametrize("B,lens,cap,H,D,dtype", CASES)
def test_seq_to_head_and_back_bit_exact(B, lens, cap, H, D, dtype):
    full, x = _shards(B, lens, cap, H, D, dtype, 11)
    xd = x.to(DEV)
    y = uaa.seq_to_head(xd, lens)
    back = torch.full_like(xd, float("nan"))  # padding must be overwritten with zeros
    uaa.head_to_seq(y, lens, cap, H, out=back)
    uaa.check_device_status()
    xb = bits(x)
    np.testing.assert_array_equal(bits(y), oracle.seq_to_head(xb, lens, cap))
    np.testing.assert_array_equal(bits(back), oracle.head_to_seq(oracle.seq_to_head(xb, lens, cap), lens, cap, H))
    np.testing.assert_array_equal(bits(back), xb)  # round trip, padding rows zero
    # the head groups are the head slices of the unsharded sequence, padding heads zero
    P = len(lens)
    hg = -(-H // P)
    assert y.shape[3] == hg
    fb = bits(full)
    for g in range(P):
        real = max(0, min(hg, H - g * hg))
        np.testing.assert_array_equal(bits(y[g, :, :, :real]), fb[:, :, g * hg:g * hg + real])
        assert (bits(y[g, :, :, real:]) == 0).all()


def test_head_to_seq_of_arbitrary_groups_matches_oracle():
    lens, cap, B, H, D = (6, 2, 5, 0), 7, 2, 8, 64
    g = torch.Generator().manual_seed(3)
    y = torch.randn((4, B, sum(lens), H // 4, D), generator=g).to(torch.bfloat16)
    out = uaa.head_to_seq(y.to(DEV), lens, cap)
    np.testing.assert_array_equal(bits(out), oracle.head_to_seq(bits(y), lens, cap))


@pytest.mark.parametrize("lens,cap,B", [((6821, 6821, 6819, 6819), 6821, 4), ((3, 1), 3, 1), ((0, 5, 2), 6, 3)])
def test_assemble_key_mask_bit_exact(lens, cap, B):
    g = torch.Generator().manual_seed(5)
    gathered = (torch.rand((len(lens), B, cap), generator=g) < 0.6).to(torch.uint8)
    m = uaa.assemble_key_mask(gathered.to(DEV), lens)
    np.testing.assert_array_equal(m.cpu().numpy(), oracle.assemble_key_mask(gathered.numpy(), lens))
    # and the result is never the untrimmed concatenation when shards are uneven
    if len(set(lens)) > 1:
        assert m.shape[1] != oracle.assemble_key_mask_untrimmed(gathered.numpy()).shape[1]


def test_assemble_key_mask_from_split_prefix_mask():
    w = synth.workload("ulysses_p4_n27280_h40_d128")
    lens = w.shard_lens
    mask = (torch.arange(w.S)[None, :] < 20000).to(torch.uint8)
    gathered = torch.from_numpy(oracle.split_key_mask(mask.numpy(), lens, w.cap))
    m = uaa.assemble_key_mask(gathered.to(DEV), lens)
    assert torch.equal(m.cpu(), mask)
