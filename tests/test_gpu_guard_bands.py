"""Out-of-bounds writes: every output of the attention calls is placed inside a
larger device buffer whose bytes before and after it hold a canary pattern; after
the call every canary byte must be unchanged.  Ragged sequence lengths (partial
last tiles, a single row) and the Ulysses path with eight shards of uneven
length (tiles that end inside each shard) are the cases where a kernel could
write past a tensor's end.  This stands in for a memory checker, which is not
available on this GPU pool."""
import math

import pytest
import torch

import ulysses_dit_attention_gb300 as uaa
from ulysses_dit_attention_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"
CANARY = 0xA5
GUARD = 8192  # bytes on each side (keeps 256-byte alignment)


class Guarded:
    def __init__(self):
        self.bufs = []

    def empty(self, shape, dtype):
        n = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        buf = torch.full((n + 2 * GUARD,), CANARY, dtype=torch.uint8, device=DEV)
        self.bufs.append((buf, n))
        return buf[GUARD:GUARD + n].view(dtype).view(shape)

    def check(self):
        torch.cuda.synchronize()
        for buf, n in self.bufs:
            head, tail = buf[:GUARD], buf[GUARD + n:]
            assert bool((head == CANARY).all()), "write before the start of an output"
            assert bool((tail == CANARY).all()), "write past the end of an output"


@pytest.mark.parametrize("S", [1, 127, 129, 257])
@pytest.mark.parametrize("D,masked", [(128, False), (64, True), (128, True)])
def test_attention_writes_stay_inside_their_outputs(S, D, masked):
    B, H = 2, 3
    inp = synth.draw(B, S, H, D, seed=S * 3 + D, masked=masked)
    q, k, v, do = (inp[n].to(DEV) for n in ("q", "k", "v", "do"))
    mask = None if inp["mask"] is None else inp["mask"].to(DEV)
    scale = 1.0 / math.sqrt(D)
    g = Guarded()
    out = g.empty((B, S, H, D), torch.bfloat16)
    lse = g.empty((B, H, S), torch.float32)
    uaa.attn_fwd(q, k, v, mask, scale, out=out, lse=lse)
    dq, dk, dv = (g.empty((B, S, H, D), torch.bfloat16) for _ in range(3))
    ws = g.empty((uaa.attn_bwd_workspace_bytes(B, S, H, D),), torch.uint8)
    uaa.attn_bwd(q, k, v, out, do, lse, mask, scale, dq=dq, dk=dk, dv=dv, workspace=ws)
    uaa.check_device_status()
    g.check()
    assert torch.isfinite(out.float()).all() and torch.isfinite(dq.float()).all()


@pytest.mark.parametrize("D", [64, 128])
def test_fused_ulysses_writes_stay_inside_their_outputs(D):
    lens, cap, B, H = (50, 33, 50, 50, 33, 50, 0, 33), 64, 2, 2
    N = sum(lens)
    inp = synth.draw(B, N, H, D, seed=88 + D)
    sh = {n: synth.pad_shards(inp[n], lens, cap).to(DEV) for n in ("q", "k", "v", "do")}
    g = Guarded()
    shape = (len(lens), B, cap, H, D)
    o = g.empty(shape, torch.bfloat16)
    lse = g.empty((B, H, N), torch.float32)
    uaa.ulysses_attn_fwd(sh["q"], sh["k"], sh["v"], lens, None, None, out=o, lse=lse)
    dq, dk, dv = (g.empty(shape, torch.bfloat16) for _ in range(3))
    ws = g.empty((uaa.ulysses_attn_bwd_workspace_bytes(lens, cap, B, H, D),), torch.uint8)
    uaa.ulysses_attn_bwd(sh["q"], sh["k"], sh["v"], o, sh["do"], lse, lens, None, None, dq=dq, dk=dk, dv=dv,
                         workspace=ws)
    uaa.check_device_status()
    g.check()


def test_relayout_writes_stay_inside_their_outputs():
    lens, cap, B, H, D = (301, 300, 257, 130), 301, 2, 6, 128
    x = synth.pad_shards(synth.draw(B, sum(lens), H, D, seed=5, with_grad_out=False)["q"], lens, cap).to(DEV)
    g = Guarded()
    y = g.empty((4, B, sum(lens), 2, D), torch.bfloat16)
    uaa.seq_to_head(x, lens, out=y)
    back = g.empty(tuple(x.shape), torch.bfloat16)
    uaa.head_to_seq(y, lens, cap, H, out=back)
    gathered = (torch.rand((4, B, cap)) < 0.5).to(torch.uint8).to(DEV)
    m = g.empty((B, sum(lens)), torch.uint8)
    uaa.assemble_key_mask(gathered, lens, out=m)
    uaa.check_device_status()
    g.check()
    assert torch.equal(back.view(torch.int16), x.view(torch.int16))
