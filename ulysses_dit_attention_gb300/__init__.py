"""GB300-native Ulysses DiT attention: thin Python binding over the ``libuaa.so`` C ABI.

Every step of the computation runs in the library's sm_103a kernels; this module
only marshals arguments (shapes, dtypes, pointers, the current CUDA stream) and
allocates outputs/workspace with PyTorch.  There is no CPU or eager fallback: if
the library is not built, or the tensors are not on a CUDA device, calls raise.

Names follow the C ABI (``include/uaa.h``): ``attn_fwd``, ``attn_bwd``,
``seq_to_head``, ``head_to_seq``, ``assemble_key_mask``; ``Attention`` is the
``torch.autograd.Function`` pairing them (the LSE output is marked
non-differentiable, as in "[attention] Add Ulysses Anything backward", What does
this PR do), and ``ulysses_attention`` composes the Ulysses exchange around it
for P emulated ranks on one device.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from .build import DEBUG_LIB_PATH, LIB_PATH

__all__ = [
    "UAAError", "lib", "attn_fwd", "attn_bwd", "attn_bwd_workspace_bytes", "attn_bwd_fused_workspace_bytes", "seq_to_head", "head_to_seq",
    "assemble_key_mask", "check_device_status", "watchdog_selftest", "set_wait_timeout_ms", "debug_drop_load",
    "set_bwd_profile_events", "Attention", "attn_fwd_groups", "attn_bwd_groups",
    "attention", "UlyssesAttention", "ulysses_attention", "STATUS", "debug_build", "debug_exp2_fma2",
]

STATUS = {0: "UAA_OK", -1: "UAA_ERR_INVALID_ARG", -2: "UAA_ERR_UNSUPPORTED", -3: "UAA_ERR_PER_HEAD_MASK",
          -4: "UAA_ERR_CUDA", -5: "UAA_ERR_TIMEOUT", -6: "UAA_ERR_DEBUG_CHECK"}


class UAAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


_lib = None
_lib_lock = threading.Lock()

_P = ctypes.c_void_p
_I = ctypes.c_int
_SIGS = {
    "uaa_attn_fwd": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, ctypes.c_float, _P]),
    "uaa_attn_fwd_cross": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_float, _P]),
    "uaa_attn_bwd_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "uaa_attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, ctypes.c_float, _P,
                          ctypes.c_size_t, _P]),
    "uaa_attn_bwd_cross": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_float, _P,
                                ctypes.c_size_t, _P]),
    "uaa_attn_bwd_fused_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "uaa_attn_bwd_fused": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, ctypes.c_float, _P,
                                ctypes.c_size_t, _P]),
    "uaa_attn_fwd_groups": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_float, _P]),
    "uaa_attn_bwd_groups": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_float, _P,
                                 ctypes.c_size_t, _P]),
    "uaa_attn_bwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, ctypes.c_float, _P]),
    "uaa_attn_bwd_noalloc_max_bytes": (ctypes.c_size_t, []),
    "uaa_ulysses_attn_fwd": (_I, [_P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, ctypes.c_float, _P]),
    "uaa_ulysses_attn_bwd_workspace_bytes": (ctypes.c_size_t, [_I, _P, _I, _I, _I, _I]),
    "uaa_ulysses_attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, ctypes.c_float,
                                  _P, ctypes.c_size_t, _P]),
    "uaa_seq_to_head": (_I, [_P, _P, _I, _P, _I, _I, _I, _I, _I, _P]),
    "uaa_head_to_seq": (_I, [_P, _P, _I, _P, _I, _I, _I, _I, _I, _P]),
    "uaa_assemble_key_mask": (_I, [_P, _P, _I, _P, _I, _I, _P]),
    "uaa_check_device_status": (_I, [_P]),
    "uaa_watchdog_selftest": (_I, [ctypes.c_uint, _P]),
    "uaa_set_wait_timeout_ms": (None, [ctypes.c_uint]),
    "uaa_debug_drop_load": (None, [_I]),
    "uaa_set_bwd_profile_events": (None, [_P, _P, _P]),
    "uaa_last_error": (ctypes.c_char_p, []),
    "uaa_version": (ctypes.c_char_p, []),
    "uaa_debug_build": (_I, []),
    "uaa_debug_exp2_fma2": (_I, [_P, _P, ctypes.c_longlong, _P]),
}


def lib():
    """Load ``libuaa.so`` (once; ``libuaa_debug.so``, the build with device range checks,
    when the environment sets ``UAA_DEBUG=1``).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        with _lib_lock:
            if _lib is None:
                debug = os.environ.get("UAA_DEBUG", "") == "1"
                path = DEBUG_LIB_PATH if debug else LIB_PATH
                if not os.path.exists(path):
                    how = "--debug " if debug else ""
                    raise RuntimeError(f"{path} is missing: build it with "
                                       f"`python -m ulysses_dit_attention_gb300.build {how}` (no fallback exists)")
                handle = ctypes.CDLL(path)
                for name, (res, args) in _SIGS.items():
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


def _check(status: int):
    if status != 0:
        raise UAAError(status, lib().uaa_last_error().decode(errors="replace"))


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("uaa kernels run on CUDA tensors only (no CPU fallback)")


def _bshd(name, t, ref=None, same_s=True):
    if t.dim() != 4:
        raise ValueError(f"{name} must be (B, S, H, D), got {tuple(t.shape)}")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous BSHD")
    if ref is not None:
        a, b = tuple(t.shape), tuple(ref.shape)
        if (a != b) if same_s else (a[0] != b[0] or a[2:] != b[2:]):
            raise ValueError(f"{name} shape {a} does not fit {b}")


def normalize_key_mask(mask, B, S):
    """Key mask -> contiguous uint8 ``(B, S)``.

    Accepts ``(B, S)`` or the head-broadcast ``(B, 1, 1, S)`` form; a per-head
    ``(B, H>1, 1, S)`` mask raises ``ValueError`` before any launch ("[attention]
    Add Ulysses Anything backward", What does this PR do: fail fast on per-head
    masks, which Ulysses cannot shard).  A bool mask is reinterpreted as bytes
    (no copy kernel).
    """
    if mask is None:
        return None
    if mask.dim() == 4:
        if mask.shape[1] != 1 or mask.shape[2] != 1:
            raise ValueError(f"per-head attention masks {tuple(mask.shape)} are not supported: only "
                             "head-broadcast (B, 1, 1, S) key masks can be sharded across heads")
        mask = mask.reshape(mask.shape[0], mask.shape[3])
    if mask.dim() != 2 or tuple(mask.shape) != (B, S):
        raise ValueError(f"key mask must be (B, S) = {(B, S)}, got {tuple(mask.shape)}")
    if mask.dtype == torch.bool:
        mask = mask.view(torch.uint8)
    if mask.dtype != torch.uint8:
        raise TypeError("key mask must be bool or uint8")
    if not mask.is_contiguous():
        raise ValueError("key mask must be contiguous")
    return mask


# --------------------------------------------------------------------------- attention
def attn_fwd(q, k, v, key_mask=None, scale=None, out=None, lse=None):
    """``uaa_attn_fwd`` / ``uaa_attn_fwd_cross``: returns ``(out bf16 (B,Sq,H,D), lse fp32 (B,H,Sq))``.

    ``k`` and ``v`` may have another sequence length ``Sk`` than ``q`` (cross-attention);
    ``key_mask`` is then ``(B, Sk)``.
    """
    _bshd("q", q)
    _bshd("k", k, q, same_s=False)
    _bshd("v", v, k)
    _need_cuda(q, k, v)
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    mask = normalize_key_mask(key_mask, B, Sk)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    if Sq == Sk:
        _check(lib().uaa_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(mask), _ptr(out), _ptr(lse), B, Sq, H, D,
                                  float(scale), _P(_stream(q.device))))
    else:
        _check(lib().uaa_attn_fwd_cross(_ptr(q), _ptr(k), _ptr(v), _ptr(mask), _ptr(out), _ptr(lse), B, Sq, Sk, H,
                                        D, float(scale), _P(_stream(q.device))))
    return out, lse


def attn_bwd_workspace_bytes(B, S, H, D) -> int:
    return int(lib().uaa_attn_bwd_workspace_bytes(B, S, H, D))


def attn_bwd_fused_workspace_bytes(B, S, H, D) -> int:
    return int(lib().uaa_attn_bwd_fused_workspace_bytes(B, S, H, D))


def attn_bwd(q, k, v, out, dout, lse, key_mask=None, scale=None, dq=None, dk=None, dv=None, workspace=None,
             fused=False):
    """``uaa_attn_bwd`` / ``uaa_attn_bwd_cross``: returns ``(dq, dk, dv)`` in bf16 BSHD.

    ``k``, ``v`` (and ``dk``, ``dv``) may have another sequence length than ``q``.  With
    ``fused=True`` (same sequence lengths only) the one-pass ``uaa_attn_bwd_fused`` runs
    instead: five GEMMs instead of seven, dQ by fp32 reductions, so dQ is not bit-for-bit
    reproducible.
    """
    _bshd("q", q)
    _bshd("k", k, q, same_s=False)
    _bshd("v", v, k)
    _bshd("out", out, q)
    _bshd("dout", dout, q)
    _need_cuda(q, k, v, out, dout, lse)
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, Sq) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 (B, H, Sq)")
    mask = normalize_key_mask(key_mask, B, Sk)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(k) if dv is None else dv
    if fused and Sq != Sk:
        raise ValueError("the fused backward takes equal query and key lengths")
    nbytes = attn_bwd_fused_workspace_bytes(B, Sq, H, D) if fused else attn_bwd_workspace_bytes(B, Sq, H, D)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    wsb = workspace.numel() * workspace.element_size()
    if fused:
        _check(lib().uaa_attn_bwd_fused(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(mask),
                                        _ptr(dq), _ptr(dk), _ptr(dv), B, Sq, H, D, float(scale), _ptr(workspace), wsb,
                                        _P(_stream(q.device))))
    elif Sq == Sk:
        _check(lib().uaa_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(mask),
                                  _ptr(dq), _ptr(dk), _ptr(dv), B, Sq, H, D, float(scale), _ptr(workspace), wsb,
                                  _P(_stream(q.device))))
    else:
        _check(lib().uaa_attn_bwd_cross(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(mask),
                                        _ptr(dq), _ptr(dk), _ptr(dv), B, Sq, Sk, H, D, float(scale),
                                        _ptr(workspace), wsb, _P(_stream(q.device))))
    return dq, dk, dv


def _groups(name, t, ref=None):
    if t.dim() != 5:
        raise ValueError(f"{name} must be (G, B, S, H, D), got {tuple(t.shape)}")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (G, B, S, H, D)")
    if ref is not None and tuple(t.shape) != tuple(ref.shape):
        raise ValueError(f"{name} shape {tuple(t.shape)} does not fit {tuple(ref.shape)}")


def attn_fwd_groups(q, k, v, key_mask=None, scale=None, out=None, lse=None):
    """``uaa_attn_fwd_groups``: attention of G head groups ``(G, B, S, H, D)`` in one launch.

    The ``(B, S)`` key mask is shared by the G groups.  Returns ``(out, lse)`` with ``lse``
    fp32 ``(G, B, H, S)``.
    """
    _groups("q", q)
    _groups("k", k, q)
    _groups("v", v, q)
    _need_cuda(q, k, v)
    G, B, S, H, D = q.shape
    mask = normalize_key_mask(key_mask, B, S)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((G, B, H, S), dtype=torch.float32, device=q.device)
    _check(lib().uaa_attn_fwd_groups(_ptr(q), _ptr(k), _ptr(v), _ptr(mask), _ptr(out), _ptr(lse), G, B, S, H, D,
                                     float(scale), _P(_stream(q.device))))
    return out, lse


def attn_bwd_groups(q, k, v, out, dout, lse, key_mask=None, scale=None, dq=None, dk=None, dv=None, workspace=None):
    """``uaa_attn_bwd_groups``: the backward of :func:`attn_fwd_groups`; returns ``(dq, dk, dv)``."""
    for n, t in (("k", k), ("v", v), ("out", out), ("dout", dout)):
        _groups(n, t, q)
    _groups("q", q)
    _need_cuda(q, k, v, out, dout, lse)
    G, B, S, H, D = q.shape
    if lse.dtype != torch.float32 or tuple(lse.shape) != (G, B, H, S) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 (G, B, H, S)")
    mask = normalize_key_mask(key_mask, B, S)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    nbytes = attn_bwd_workspace_bytes(G * B, S, H, D)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    wsb = workspace.numel() * workspace.element_size()
    _check(lib().uaa_attn_bwd_groups(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(mask),
                                     _ptr(dq), _ptr(dk), _ptr(dv), G, B, S, H, D, float(scale), _ptr(workspace), wsb,
                                     _P(_stream(q.device))))
    return dq, dk, dv


class Attention(torch.autograd.Function):
    """Autograd pairing of ``attn_fwd`` / ``attn_bwd``; ``lse`` is non-differentiable."""

    @staticmethod
    def forward(ctx, q, k, v, key_mask=None, scale=None):
        out, lse = attn_fwd(q, k, v, key_mask, scale)
        ctx.save_for_backward(q, k, v, out, lse)
        ctx.key_mask = key_mask
        ctx.scale = scale
        ctx.mark_non_differentiable(lse)
        return out, lse

    @staticmethod
    def backward(ctx, dout, _dlse):
        q, k, v, out, lse = ctx.saved_tensors
        dq, dk, dv = attn_bwd(q, k, v, out, dout.contiguous(), lse, ctx.key_mask, ctx.scale)
        return dq, dk, dv, None, None


def attention(q, k, v, key_mask=None, scale=None):
    return Attention.apply(q, k, v, key_mask, scale)


# --------------------------------------------------------------------------- Ulysses re-layout
def _lens_array(shard_lens):
    lens = [int(x) for x in shard_lens]
    return (ctypes.c_int * len(lens))(*lens), lens


def seq_to_head(x, shard_lens, out=None):
    """``uaa_seq_to_head``: ``(P, B, cap, H, D)`` shards -> ``(P, B, N, ceil(H/P), D)`` groups.

    When P does not divide H the groups are padded with zero heads.
    """
    _need_cuda(x)
    if x.dim() != 5 or not x.is_contiguous():
        raise ValueError("x must be contiguous (P, B, cap, H, D)")
    P, B, cap, H, D = x.shape
    arr, lens = _lens_array(shard_lens)
    if len(lens) != P:
        raise ValueError("len(shard_lens) must equal P")
    N = sum(lens)
    if out is None:
        out = torch.empty((P, B, N, -(-H // P), D), dtype=x.dtype, device=x.device)
    _check(lib().uaa_seq_to_head(_ptr(x), _ptr(out), P, arr, cap, B, H, D, x.element_size(), _P(_stream(x.device))))
    return out


def head_to_seq(y, shard_lens, cap, H=None, out=None):
    """``uaa_head_to_seq``: ``(P, B, N, Hg, D)`` groups -> ``(P, B, cap, H, D)`` shards (padding zeroed).

    ``H`` is the true head count (default ``P * Hg``); padding heads of the groups are dropped.
    """
    _need_cuda(y)
    if y.dim() != 5 or not y.is_contiguous():
        raise ValueError("y must be contiguous (P, B, N, Hg, D)")
    P, B, N, Hg, D = y.shape
    H = P * Hg if H is None else int(H)
    if not (Hg - 1) * P < H <= Hg * P:
        raise ValueError(f"H={H} does not have ceil(H/P) = {Hg} heads per group")
    arr, lens = _lens_array(shard_lens)
    if len(lens) != P or sum(lens) != N:
        raise ValueError("shard_lens must have P entries summing to N")
    if out is None:
        out = torch.empty((P, B, cap, H, D), dtype=y.dtype, device=y.device)
    _check(lib().uaa_head_to_seq(_ptr(y), _ptr(out), P, arr, cap, B, H, D, y.element_size(),
                                 _P(_stream(y.device))))
    return out


def assemble_key_mask(gathered, shard_lens, out=None):
    """``uaa_assemble_key_mask``: gathered ``(P, B, cap)`` uint8 -> trimmed ``(B, N)`` uint8."""
    _need_cuda(gathered)
    if gathered.dtype == torch.bool:
        gathered = gathered.view(torch.uint8)
    if gathered.dim() != 3 or gathered.dtype != torch.uint8 or not gathered.is_contiguous():
        raise ValueError("gathered must be contiguous uint8 (P, B, cap)")
    P, B, cap = gathered.shape
    arr, lens = _lens_array(shard_lens)
    if len(lens) != P:
        raise ValueError("len(shard_lens) must equal P")
    if out is None:
        out = torch.empty((B, sum(lens)), dtype=torch.uint8, device=gathered.device)
    _check(lib().uaa_assemble_key_mask(_ptr(gathered), _ptr(out), P, arr, cap, B, _P(_stream(gathered.device))))
    return out


def debug_exp2_fma2(x):
    """``uaa_debug_exp2_fma2``: the forward's FMA-pipe 2^x on a contiguous float32 CUDA tensor
    with an even number of elements (a diagnostic for tests)."""
    _need_cuda(x)
    if x.dtype != torch.float32 or not x.is_contiguous() or x.numel() % 2:
        raise ValueError("x must be a contiguous float32 tensor with an even number of elements")
    y = torch.empty_like(x)
    _check(lib().uaa_debug_exp2_fma2(_ptr(x), _ptr(y), x.numel(), _P(_stream(x.device))))
    return y


def debug_build() -> bool:
    """True when the loaded library is the debug build (device range checks)."""
    return bool(lib().uaa_debug_build())


def check_device_status(device=None):
    dev = torch.device("cuda") if device is None else torch.device(device)
    _check(lib().uaa_check_device_status(_P(_stream(dev))))


def watchdog_selftest(timeout_us=2000, device=None):
    dev = torch.device("cuda") if device is None else torch.device(device)
    return lib().uaa_watchdog_selftest(int(timeout_us), _P(_stream(dev)))


def set_wait_timeout_ms(ms: int):
    lib().uaa_set_wait_timeout_ms(int(ms))



def debug_drop_load(n: int):
    """Diagnostic: the attention kernels' producers skip their n-th ring load (-1: off)."""
    lib().uaa_debug_drop_load(int(n))


def set_bwd_profile_events(events=None):
    """Record three ``torch.cuda.Event``s around the backward's dK/dV and dQ kernels (None stops)."""
    if events is None:
        lib().uaa_set_bwd_profile_events(None, None, None)
    else:
        a, b, c = (_P(e.cuda_event) for e in events)
        lib().uaa_set_bwd_profile_events(a, b, c)


# --------------------------------------------------------------------------- Ulysses composition
class UlyssesAttention(torch.autograd.Function):
    """Ulysses attention over P emulated ranks on one device.

    Forward: seq->head exchange of Q, K, V; attention per head group (all groups
    share the assembled key mask); head->seq exchange of O.  Backward: seq->head
    exchange of dO; attention backward per group; head->seq exchange of dQ
    (query partition) and dK, dV (key partition).  "[attention] Add Ulysses
    Anything backward", What does this PR do.
    """

    @staticmethod
    def forward(ctx, q_sh, k_sh, v_sh, shard_lens, key_mask=None, scale=None):
        cap, H = q_sh.shape[2], q_sh.shape[3]
        yq, yk, yv = (seq_to_head(t, shard_lens) for t in (q_sh, k_sh, v_sh))
        P = yq.shape[0]
        # the P groups form one batch of P*B sequences sharing the B mask rows: one launch for all
        # emulated ranks
        o, lse = attn_fwd_groups(yq, yk, yv, key_mask, scale)
        o_sh = head_to_seq(o, shard_lens, cap, H)
        ctx.save_for_backward(yq, yk, yv, o, lse)
        ctx.shard_lens, ctx.key_mask, ctx.scale, ctx.cap, ctx.H = tuple(shard_lens), key_mask, scale, cap, H
        ctx.mark_non_differentiable(lse)
        return o_sh, lse

    @staticmethod
    def backward(ctx, do_sh, _dlse):
        yq, yk, yv, o, lse = ctx.saved_tensors
        ydo = seq_to_head(do_sh.contiguous(), ctx.shard_lens)
        dq, dk, dv = attn_bwd_groups(yq, yk, yv, o, ydo, lse, ctx.key_mask, ctx.scale)
        return (head_to_seq(dq, ctx.shard_lens, ctx.cap, ctx.H), head_to_seq(dk, ctx.shard_lens, ctx.cap, ctx.H),
                head_to_seq(dv, ctx.shard_lens, ctx.cap, ctx.H), None, None, None)


def ulysses_attention(q_sh, k_sh, v_sh, shard_lens, key_mask=None, scale=None):
    return UlyssesAttention.apply(q_sh, k_sh, v_sh, tuple(shard_lens), key_mask, scale)


# --------------------------------------------------------------------------- Ulysses, exchanges fused
def _shards(name, t, ref=None):
    if t.dim() != 5:
        raise ValueError(f"{name} must be (P, B, cap, H, D), got {tuple(t.shape)}")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (P, B, cap, H, D)")
    if ref is not None and tuple(t.shape) != tuple(ref.shape):
        raise ValueError(f"{name} shape {tuple(t.shape)} does not fit {tuple(ref.shape)}")


def ulysses_attn_fwd(q_sh, k_sh, v_sh, shard_lens, key_mask=None, scale=None, out=None, lse=None):
    """``uaa_ulysses_attn_fwd``: Ulysses attention straight on the sequence shards.

    ``q_sh``, ``k_sh``, ``v_sh``: ``(P, B, cap, H, D)`` bf16 shards; returns ``(out_sh, lse)`` with
    ``out_sh`` in the same layout (padding rows zero) and ``lse`` fp32 ``(B, H, N)`` in sequence
    order, N = sum(shard_lens).  ``key_mask`` is ``(B, N)`` in sequence order.
    """
    _shards("q_sh", q_sh)
    _shards("k_sh", k_sh, q_sh)
    _shards("v_sh", v_sh, q_sh)
    _need_cuda(q_sh, k_sh, v_sh)
    P, B, cap, H, D = q_sh.shape
    arr, lens = _lens_array(shard_lens)
    if len(lens) != P:
        raise ValueError("len(shard_lens) must equal P")
    N = sum(lens)
    mask = normalize_key_mask(key_mask, B, N)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q_sh)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q_sh.device)
    _check(lib().uaa_ulysses_attn_fwd(_ptr(q_sh), _ptr(k_sh), _ptr(v_sh), _ptr(mask), _ptr(out), _ptr(lse), P, arr,
                                      cap, B, H, D, float(scale), _P(_stream(q_sh.device))))
    return out, lse


def ulysses_attn_bwd_workspace_bytes(shard_lens, cap, B, H, D) -> int:
    arr, lens = _lens_array(shard_lens)
    return int(lib().uaa_ulysses_attn_bwd_workspace_bytes(len(lens), arr, cap, B, H, D))


def ulysses_attn_bwd(q_sh, k_sh, v_sh, out_sh, dout_sh, lse, shard_lens, key_mask=None, scale=None, dq=None,
                     dk=None, dv=None, workspace=None):
    """``uaa_ulysses_attn_bwd``: the backward of :func:`ulysses_attn_fwd` on the shards."""
    for n, t in (("k_sh", k_sh), ("v_sh", v_sh), ("out_sh", out_sh), ("dout_sh", dout_sh)):
        _shards(n, t, q_sh)
    _shards("q_sh", q_sh)
    _need_cuda(q_sh, k_sh, v_sh, out_sh, dout_sh, lse)
    P, B, cap, H, D = q_sh.shape
    arr, lens = _lens_array(shard_lens)
    if len(lens) != P:
        raise ValueError("len(shard_lens) must equal P")
    N = sum(lens)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 (B, H, N)")
    mask = normalize_key_mask(key_mask, B, N)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q_sh) if dq is None else dq
    dk = torch.empty_like(q_sh) if dk is None else dk
    dv = torch.empty_like(q_sh) if dv is None else dv
    nbytes = ulysses_attn_bwd_workspace_bytes(lens, cap, B, H, D)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q_sh.device)
    wsb = workspace.numel() * workspace.element_size()
    _check(lib().uaa_ulysses_attn_bwd(_ptr(q_sh), _ptr(k_sh), _ptr(v_sh), _ptr(out_sh), _ptr(dout_sh), _ptr(lse),
                                      _ptr(mask), _ptr(dq), _ptr(dk), _ptr(dv), P, arr, cap, B, H, D, float(scale),
                                      _ptr(workspace), wsb, _P(_stream(q_sh.device))))
    return dq, dk, dv


class FusedUlyssesAttention(torch.autograd.Function):
    """Ulysses attention with the exchanges fused into the attention kernels (same result as
    :class:`UlyssesAttention` up to rounding; ``lse`` is ``(B, H, N)``, non-differentiable)."""

    @staticmethod
    def forward(ctx, q_sh, k_sh, v_sh, shard_lens, key_mask=None, scale=None):
        out, lse = ulysses_attn_fwd(q_sh, k_sh, v_sh, shard_lens, key_mask, scale)
        ctx.save_for_backward(q_sh, k_sh, v_sh, out, lse)
        ctx.shard_lens, ctx.key_mask, ctx.scale = tuple(shard_lens), key_mask, scale
        ctx.mark_non_differentiable(lse)
        return out, lse

    @staticmethod
    def backward(ctx, dout, _dlse):
        q_sh, k_sh, v_sh, out, lse = ctx.saved_tensors
        dq, dk, dv = ulysses_attn_bwd(q_sh, k_sh, v_sh, out, dout.contiguous(), lse, ctx.shard_lens, ctx.key_mask,
                                      ctx.scale)
        return dq, dk, dv, None, None, None


def ulysses_attention_fused(q_sh, k_sh, v_sh, shard_lens, key_mask=None, scale=None):
    return FusedUlyssesAttention.apply(q_sh, k_sh, v_sh, tuple(shard_lens), key_mask, scale)
