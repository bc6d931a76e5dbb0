"""The C-ABI library on the CPU: it builds, loads, exports every symbol that
``include/uaa.h`` declares, and rejects bad arguments on the host before any
CUDA call (so these run without a GPU)."""
import ctypes
import os
import re

import pytest

import ulysses_dit_attention_gb300 as uaa
from ulysses_dit_attention_gb300 import build as uaa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    uaa_build.build()
    return uaa.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "uaa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(uaa_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n
    assert L.uaa_version().decode().startswith("uaa")


def test_workspace_bytes(L):
    B, S, H, D = 1, 27280, 40, 128
    got = L.uaa_attn_bwd_workspace_bytes(B, S, H, D)
    s_pad = (S + 127) // 128 * 128
    assert got == (B * H * s_pad * 8 + 255) // 256 * 256  # fp32 Delta and -LSE*log2e, rows padded to 128
    assert L.uaa_attn_bwd_workspace_bytes(1, 16, 2, 96) == 0


def _err():
    return uaa.lib().uaa_last_error().decode()


def test_attn_fwd_rejects_bad_args_on_host(L):
    P = ctypes.c_void_p
    fake = P(1 << 20)
    st = L.uaa_attn_fwd(fake, fake, fake, None, fake, fake, 1, 16, 2, 96, ctypes.c_float(0.1), None)
    assert st == -2 and "D=96" in _err()
    st = L.uaa_attn_fwd(fake, fake, fake, None, fake, fake, 1, 16, 2, 64, ctypes.c_float(-1.0), None)
    assert st == -1 and "scale" in _err()
    st = L.uaa_attn_fwd(None, fake, fake, None, fake, fake, 1, 16, 2, 64, ctypes.c_float(0.125), None)
    assert st == -1 and "q is NULL" in _err()
    st = L.uaa_attn_fwd(P((1 << 20) + 8), fake, fake, None, fake, fake, 1, 16, 2, 64, ctypes.c_float(0.125), None)
    assert st == -1 and "aligned" in _err()
    # empty input: nothing to do, nothing launched
    assert L.uaa_attn_fwd(None, None, None, None, None, None, 0, 16, 2, 64, ctypes.c_float(0.125), None) == 0
    assert L.uaa_attn_fwd(None, None, None, None, None, None, 2, 0, 2, 64, ctypes.c_float(0.125), None) == 0


def test_attn_bwd_rejects_small_workspace(L):
    P = ctypes.c_void_p
    fake = P(1 << 20)
    ws = P(1 << 24)
    st = L.uaa_attn_bwd(fake, fake, fake, fake, fake, fake, None, fake, fake, fake, 1, 256, 2, 64,
                        ctypes.c_float(0.125), ws, 16, None)
    assert st == -1 and "workspace" in _err()
    st = L.uaa_attn_bwd(fake, fake, fake, fake, fake, fake, None, fake, fake, fake, 1, 256, 2, 64,
                        ctypes.c_float(0.125), P((1 << 24) + 16), 1 << 30, None)
    assert st == -1 and "256-byte" in _err()


def test_relayout_rejects_bad_partitions_on_host(L):
    P = ctypes.c_void_p
    fake = P(1 << 20)
    lens = (ctypes.c_int * 4)(6821, 6821, 6819, 6819)
    # P outside [1, 64]
    assert L.uaa_seq_to_head(fake, fake, 0, lens, 6821, 1, 40, 128, 2, None) == -1
    # a shard longer than the capacity
    assert L.uaa_seq_to_head(fake, fake, 4, lens, 6820, 1, 40, 128, 2, None) == -1
    assert "cap" in _err()
    # D * elem_bytes not a multiple of 16
    assert L.uaa_head_to_seq(fake, fake, 4, lens, 6821, 1, 40, 4, 2, None) == -1
    # negative shard length
    bad = (ctypes.c_int * 2)(3, -1)
    assert L.uaa_assemble_key_mask(fake, fake, 2, bad, 3, 1, None) == -1
    assert L.uaa_watchdog_selftest(0, None) == -1


def test_cross_attention_rejects_missing_sides_on_host(L):
    fake = ctypes.c_void_p(1 << 20)
    # queries without keys
    assert L.uaa_attn_fwd_cross(fake, fake, fake, None, fake, fake, 1, 128, 0, 2, 128, ctypes.c_float(0.1),
                                None) == -1
    assert "Sk" in _err()
    # keys without queries in the backward
    assert L.uaa_attn_bwd_cross(fake, fake, fake, fake, fake, fake, None, fake, fake, fake, 1, 0, 128, 2, 128,
                                ctypes.c_float(0.1), fake, 1 << 20, None) == -1
    assert "Sq" in _err()
    # nothing to do: no queries in the forward
    assert L.uaa_attn_fwd_cross(fake, fake, fake, None, fake, fake, 1, 0, 128, 2, 128, ctypes.c_float(0.1),
                                None) == 0


def test_python_binding_rejects_per_head_mask_before_launch():
    import torch
    with pytest.raises(ValueError, match="per-head"):
        uaa.normalize_key_mask(torch.ones(2, 4, 1, 16, dtype=torch.bool), 2, 16)
    m = uaa.normalize_key_mask(torch.ones(2, 1, 1, 16, dtype=torch.bool), 2, 16)
    assert m.dtype == torch.uint8 and tuple(m.shape) == (2, 16)


def test_python_binding_refuses_cpu_tensors():
    import torch
    q = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        uaa.attn_fwd(q, q, q)


def test_fused_ulysses_rejects_bad_partitions_on_host(L):
    fake = ctypes.c_void_p(1 << 20)
    f = ctypes.c_float(0.1)
    # more shards than the fused kernels take
    lens9 = (ctypes.c_int * 9)(*([10] * 9))
    assert L.uaa_ulysses_attn_fwd(fake, fake, fake, None, fake, fake, 9, lens9, 10, 1, 2, 128, f, None) == -2
    assert "P=9" in _err()
    # a shard longer than the capacity, a negative one, no lengths at all
    bad = (ctypes.c_int * 2)(11, 5)
    assert L.uaa_ulysses_attn_fwd(fake, fake, fake, None, fake, fake, 2, bad, 10, 1, 2, 128, f, None) == -1
    neg = (ctypes.c_int * 2)(3, -1)
    assert L.uaa_ulysses_attn_bwd(fake, fake, fake, fake, fake, fake, None, fake, fake, fake, 2, neg, 10, 1, 2, 128,
                                  f, fake, 1 << 20, None) == -1
    assert L.uaa_ulysses_attn_fwd(fake, fake, fake, None, fake, fake, 2, None, 10, 1, 2, 128, f, None) == -1
    # workspace: Delta and -LSE*log2e per row of every 128-row tile, tiles never straddling shards
    ok = (ctypes.c_int * 3)(130, 1, 128)
    tiles = 2 + 1 + 1
    assert L.uaa_ulysses_attn_bwd_workspace_bytes(3, ok, 130, 2, 5, 64) == (2 * 5 * tiles * 128 * 8 + 255) // 256 * 256
    assert L.uaa_ulysses_attn_bwd_workspace_bytes(9, lens9, 10, 1, 2, 128) == 0


def test_grouped_and_one_pass_backward_validate_on_host(L):
    fake = ctypes.c_void_p(1 << 20)
    f = ctypes.c_float(0.125)
    # the grouped calls need G >= 1 and G*B <= 65535
    assert L.uaa_attn_fwd_groups(fake, fake, fake, None, fake, fake, 0, 2, 128, 2, 64, f, None) == -1
    assert "G=0" in _err()
    assert L.uaa_attn_fwd_groups(fake, fake, fake, None, fake, fake, 300, 300, 128, 2, 64, f, None) == -2
    assert L.uaa_attn_bwd_groups(fake, fake, fake, fake, fake, fake, None, fake, fake, fake, 4, 2, 128, 2, 64, f,
                                 fake, 16, None) == -1
    assert "workspace" in _err()
    # grouped backward workspace: the plain backward's for a batch of G*B
    assert L.uaa_attn_bwd_workspace_bytes(8, 300, 2, 64) == (8 * 2 * 384 * 8 + 255) // 256 * 256
    # one-pass backward: the two row vectors plus an fp32 (B, H, S_pad, D) dQ accumulator
    B, S, H, D = 2, 300, 3, 128
    rows = B * H * 384
    assert L.uaa_attn_bwd_fused_workspace_bytes(B, S, H, D) == (rows * 8 + rows * D * 4 + 255) // 256 * 256
    assert L.uaa_attn_bwd_fused_workspace_bytes(B, S, H, 96) == 0
    need = L.uaa_attn_bwd_fused_workspace_bytes(B, S, H, D)
    assert L.uaa_attn_bwd_fused(fake, fake, fake, fake, fake, fake, None, fake, fake, fake, B, S, H, D, f, fake,
                                need - 256, None) == -1
    assert "workspace" in _err()
    # the diagnostic load-drop knob takes any value and is switched off by a negative one
    L.uaa_debug_drop_load(3)
    L.uaa_debug_drop_load(-1)
