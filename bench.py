"""Throughput of the Ulysses DiT attention hot path on GB300.

One step = one pass of the whole path over the Ulysses emulation workload
(B=1, N=27280 split into P=4 virtual sequence shards of 6821/6821/6819/6819
rows, H=40, D=128, bf16 N(0,1) inputs):
  seq->head exchange of Q, K, V -> attention forward of the four 10-head
  groups (O, LSE) -> head->seq exchange of O -> seq->head exchange of dO ->
  attention backward of the groups (Delta preprocess, K/V-tile-major dK/dV
  kernel, Q-tile-major dQ kernel) -> head->seq exchange of dQ, dK, dV.
The four head groups are contiguous (P, B, N, H/P, D) tensors, i.e. one BSHD
tensor of batch P*B, so each attention kernel runs once over all groups (the
work one GPU does for the four emulated ranks, in one launch).
Every step runs through the C ABI (``libuaa.so``).

``value`` = attention fwd+bwd FLOPs (4*B*H*S^2*D + 10*B*H*S^2*D) per second of
the whole step (re-layouts included), inputs resident in HBM.  The inputs
(4 x 279 MB) are larger than L2 (129 MB), so no L2 flush is added.  ``e2e``
adds, every step, the host->device copy of the step's input shards from pinned
memory and the device->host copy of O, dQ, dK, dV, on copy streams that overlap
the compute where the data dependencies allow.  ``--impl reference`` times the fp64
CPU oracle on bounded samples of the same workload instead.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from ulysses_dit_attention_gb300 import synth  # noqa: E402

WORKLOAD = "ulysses_p4_n27280_h40_d128"

# DRAM bytes (read + write) per attn_bwd_dkdv_kernel launch of the workload above (all four
# 10-head groups in one launch), from a one-pass ncu capture of the full-size launch
# (dram__bytes_read.sum 1134219008 + dram__bytes_write.sum 533566976 bytes); keyed by the
# SHA-256 prefix of the attn_bwd.cu it was taken on (re-keyed after comment-only edits of that
# file), so the bench reports null once the kernel source has changed since.
DKDV_TRAFFIC = {"e526c8e311b881bc": 1134219008 + 533566976}
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def dkdv_traffic():
    import hashlib
    src = os.path.join(ROOT, "ulysses_dit_attention_gb300", "csrc", "attn_bwd.cu")
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return DKDV_TRAFFIC.get(h)


def flops(B, S, H, D, fwd=True, bwd=True):
    f = 0
    if fwd:
        f += 4 * B * H * S * S * D
    if bwd:
        f += 10 * B * H * S * S * D
    return f


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            return d, "measured"
        except Exception:
            pass
    return dict(FALLBACK), "fallback"


def _peak_value(d, *keys):
    for k in keys:
        v = d.get(k)
        if isinstance(v, (int, float)) and v > 0:
            return float(v), k
    return None, None


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for line in (getattr(self, "out", "") or "").strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9:
                rows.append(f)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w": statistics.median(pw) if pw else None}


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, x, device="cuda"):
    """The slowest rank's time: every rank gets the maximum of ``x`` over the process group."""
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([x], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())
    return x


# --------------------------------------------------------------------------- oracle timing
def oracle_sample(inp, w, seconds=10.0, rows_per_block=512, max_blocks=None):
    """Times the fp64 oracle on query-row blocks of one head (fwd + bwd), all keys.

    Returns (flops_done, seconds_taken, description).  Rows are independent, so
    a block of query rows against all keys is a fixed fraction of the workload.
    """
    import numpy as np

    import oracle

    h = 0
    kk = inp["k"][:, :, [h]].float().numpy().astype(np.float64)
    vv = inp["v"][:, :, [h]].float().numpy().astype(np.float64)
    done = 0
    t0 = time.perf_counter()
    nblk = 0
    while True:
        r0 = (nblk * rows_per_block) % w.S
        r1 = min(w.S, r0 + rows_per_block)
        qq = inp["q"][:, r0:r1, [h]].float().numpy().astype(np.float64)
        dd = inp["do"][:, r0:r1, [h]].float().numpy().astype(np.float64)
        oracle.attn_fwd(qq, kk, vv, None, w.scale)
        oracle.attn_bwd(qq, kk, vv, dd, None, w.scale)
        done += 14 * (r1 - r0) * w.S * w.D
        nblk += 1
        el = time.perf_counter() - t0
        if el >= seconds or (max_blocks and nblk >= max_blocks):
            break
    desc = (f"fp64 NumPy oracle, fwd+bwd of {nblk} block(s) of {rows_per_block} query rows x {w.S} keys of "
            f"head {h} (D={w.D}); FLOPs counted as 14*rows*S*D")
    return done, el, desc


def cpu_cores():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        v = os.environ.get(var)
        if v and v.isdigit():
            return int(v)
    return os.cpu_count() or 1


def valid_keys(w, inp):
    """Sum over batches of the attended key count (S per batch without a mask)."""
    if inp["mask"] is None:
        return w.B * w.S
    return int(inp["mask"].to(torch.int64).sum())


def oracle_config(w, inp, seconds):
    """Times the fp64 oracle's forward + backward on workload ``w``.

    Heads are independent, so the oracle runs head by head (all batches, all
    rows) until every head is done or ``seconds`` have passed; when it stopped
    early the full time is extrapolated by the FLOPs done.  For a sequence too
    long to finish one head within the budget, blocks of query rows of one head
    are timed instead (rows are independent too).  Returns a dict for the JSON line.
    """
    import numpy as np

    import oracle

    f64 = lambda t: t.float().numpy().astype(np.float64)  # noqa: E731
    m = None if inp["mask"] is None else inp["mask"].numpy().astype(bool)
    total = 14 * w.H * w.S * w.D * valid_keys(w, inp)
    head_flops = total / w.H
    # one head of the 27280-row sequence takes ~20 s on 16 cores: sample row blocks instead
    if w.S > 8192:
        f, t, desc = oracle_sample(inp, w, seconds=seconds)
        return {"tflops": f / t / 1e12, "full_s": total / (f / t), "timed_s": t, "extrapolated": True,
                "cores": cpu_cores(), "sample": desc}
    done, heads = 0, 0
    t0 = time.perf_counter()
    for h in range(w.H):
        q, k, v, do = (f64(inp[n][:, :, [h]]) for n in ("q", "k", "v", "do"))
        oracle.attn_fwd(q, k, v, m, w.scale)
        oracle.attn_bwd(q, k, v, do, m, w.scale)
        done += head_flops
        heads += 1
        if time.perf_counter() - t0 >= seconds:
            break
    t = time.perf_counter() - t0
    full = heads == w.H
    desc = (f"fp64 NumPy oracle, fwd+bwd of {heads} of {w.H} heads (all {w.B} batches, {w.S} query rows); "
            f"FLOPs counted as 14*H*S*sum(valid keys)*D")
    return {"tflops": done / t / 1e12, "full_s": t if full else total / (done / t), "timed_s": t,
            "extrapolated": not full, "cores": cpu_cores(), "sample": desc}


# The workloads timed beside the headline: the layout trap, the 1k DiT shape, the key-padding
# mask case and the full 40-head DiT layer.  (The Ulysses emulation is the headline itself.)
PER_CONFIG = ("layout_b2_s16_h16_d64", "dit_b2_s1024_h24_d64", "mask_b4_s4096_h24_d128",
              "dit_b1_s27280_h40_d128")
L2_FLUSH_BYTES = 256 << 20  # twice the 129 MB L2


def time_config(uaa, w, dev, warmup, iters, fused_bwd=False):
    """fwd, bwd and fwd+bwd of one workload through the C ABI, each captured once in a CUDA graph
    and replayed: CUDA events around every replay, the L2 flushed (a 256 MB write) between replays
    when the inputs fit in L2, median over ``iters`` replays; plus the backward's per-kernel split
    from an eager call with the profiling events."""
    inp = synth.make(w)
    B, S, H, D = w.B, w.S, w.H, w.D
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    mask = None if inp["mask"] is None else inp["mask"].to(dev)
    out, dq, dk, dv = (torch.empty_like(q) for _ in range(4))
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    ws_fn = uaa.attn_bwd_fused_workspace_bytes if fused_bwd else uaa.attn_bwd_workspace_bytes
    ws = torch.empty(max(1, ws_fn(B, S, H, D)), dtype=torch.uint8, device=dev)
    in_bytes = 4 * q.numel() * q.element_size()
    flush = in_bytes < 2 * (129 << 20)
    scratch = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev) if flush else None

    def fwd():
        uaa.attn_fwd(q, k, v, mask, w.scale, out=out, lse=lse)

    def bwd():
        uaa.attn_bwd(q, k, v, out, do, lse, mask, w.scale, dq=dq, dk=dk, dv=dv, workspace=ws, fused=fused_bwd)

    def both():
        fwd()
        bwd()

    for _ in range(2):  # eager warm-up: loads the library, caches the device context and attributes
        both()
    torch.cuda.synchronize()
    uaa.check_device_status(dev)
    stream = torch.cuda.Stream(dev)
    graphs = {}
    for name, fn in (("fwd", fwd), ("bwd", bwd), ("fwd_bwd", both)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        graphs[name] = g
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream(dev)
    ms = {}
    for name, g in graphs.items():
        for _ in range(warmup):
            g.replay()
        times = []
        for _ in range(iters):
            if flush:
                scratch.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(cur)
            g.replay()
            e1.record(cur)
            times.append((e0, e1))
        torch.cuda.synchronize()
        ms[name] = statistics.median(a.elapsed_time(b) for a, b in times)
    # per-kernel split of the backward (eager calls, profiling events around the dK/dV and dQ kernels)
    trios = []
    for _ in range(max(3, iters // 4)):
        if flush:
            scratch.fill_(1)
        trio = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        for e in trio:  # torch only times events it has recorded itself once
            e.record(torch.cuda.current_stream(dev))
        uaa.set_bwd_profile_events(trio)
        bwd()
        uaa.set_bwd_profile_events(None)
        trios.append(trio)
    torch.cuda.synchronize()
    uaa.check_device_status(dev)
    dkdv_ms = statistics.median(a.elapsed_time(b) for a, b, _ in trios)
    dq_ms = statistics.median(b.elapsed_time(c) for _, b, c in trios)
    del graphs
    L = valid_keys(w, inp)
    ffl, bfl = 4 * H * S * D * L, 10 * H * S * D * L
    rec = {"B": B, "S": S, "H": H, "D": D, "masked": inp["mask"] is not None, "valid_keys": L,
           "fwd_ms": ms["fwd"], "bwd_ms": ms["bwd"], "fwd_bwd_ms": ms["fwd_bwd"],
           "fwd_tflops": ffl / (ms["fwd"] * 1e-3) / 1e12, "bwd_tflops": bfl / (ms["bwd"] * 1e-3) / 1e12,
           "fwd_bwd_tflops": (ffl + bfl) / (ms["fwd_bwd"] * 1e-3) / 1e12,
           "bwd_kernels_ms": ({"attn_bwd_fused_kernel": dkdv_ms, "dq_convert_kernel": dq_ms} if fused_bwd else
                              {"attn_bwd_dkdv_kernel": dkdv_ms, "attn_bwd_dq_kernel": dq_ms}),
           "bwd": "one pass, dQ by fp32 reductions" if fused_bwd else "split dK/dV and dQ passes",
           "timing": (f"CUDA graph replays, median of {iters}, "
                      + ("L2 flushed (256 MB write) before each replay" if flush else
                         "inputs larger than L2, no flush"))}
    del q, k, v, do, out, dq, dk, dv, lse, ws, scratch
    torch.cuda.empty_cache()
    return rec


def run_one_workload(args, local):
    """``--workload NAME``: the per-workload record of one workload alone (used for profiling)."""
    import ulysses_dit_attention_gb300 as uaa
    from ulysses_dit_attention_gb300 import build as uaa_build

    uaa_build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = synth.workload(args.workload)
    big = w.S * w.S * w.H * w.B > (1 << 32)
    rec = time_config(uaa, w, dev, warmup=args.warmup, iters=args.steps if big else max(args.steps, 10),
                      fused_bwd=args.bwd == "fused")
    print(json.dumps({"workload": w.name, **rec}))


def run_configs(uaa, args, dev, local):
    """One record per workload of PER_CONFIG: GPU times and fractions of the measured peaks, then the
    oracle on the host cores (after the GPU part, so the clock record covers the GPU work only)."""
    pk, src = peaks()
    sus, _ = _peak_value(pk, "bf16_tflops_sustained", "bf16_tflops")
    burst, _ = _peak_value(pk, "bf16_tflops")
    recs = {}
    with Clocks(local) as clk:
        for name in PER_CONFIG:
            w = synth.workload(name)
            # 10 warm-up and 50 timed replays of each graph, the median reported
            recs[name] = time_config(uaa, w, dev, warmup=10, iters=50, fused_bwd=args.bwd == "fused")
    for name in PER_CONFIG:
        w = synth.workload(name)
        r = recs[name]
        for key in ("fwd", "bwd", "fwd_bwd"):
            r[f"{key}_frac_sustained"] = r[f"{key}_tflops"] / sus if sus else None
            r[f"{key}_frac_burst"] = r[f"{key}_tflops"] / burst if burst else None
        if args.cpu_config_seconds > 0 and not args.no_cpu:
            r["oracle"] = oracle_config(w, synth.make(w), args.cpu_config_seconds)
    return {"workloads": recs, "peak_source": src, "peak_sustained_tflops": sus, "peak_burst_tflops": burst,
            "clocks": clk.summary()}


def run_reference(args, world, rank):
    if rank != 0:
        return
    w = synth.workload(WORKLOAD)
    inp = synth.make(w)
    times, fl = [], []
    for i in range(args.warmup + args.steps):
        f, t, desc = oracle_sample(inp, w, seconds=0.0, rows_per_block=256, max_blocks=1)
        if i >= args.warmup:
            times.append(t)
            fl.append(f)
    value = sum(fl) / sum(times) / 1e12
    line = {"metric": "attention fwd+bwd TFLOP/s", "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD, "B": w.B, "N": w.S, "P": w.P, "H": w.H, "D": w.D,
                       "shard_lens": list(w.shard_lens)},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# --------------------------------------------------------------------------- GPU arm
def run_gpu(args, world, rank, local):
    import ulysses_dit_attention_gb300 as uaa
    from ulysses_dit_attention_gb300 import build as uaa_build

    uaa_build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = synth.workload(WORKLOAD)
    workload_name = WORKLOAD
    if args.heads:
        # smaller-head variant of the same workload (same launch shapes per head group),
        # used to keep ncu captures small
        if args.heads % w.P:
            raise SystemExit("--heads must be a multiple of P=4")
        w = dataclasses.replace(w, H=args.heads)
        workload_name = f"ulysses_p4_n27280_h{args.heads}_d128"
    B, S, H, D, P = w.B, w.S, w.H, w.D, w.P
    lens, cap, Hg = w.shard_lens, w.cap, w.H // w.P
    inp = synth.make(w)
    host = {n: synth.pad_shards(inp[n], lens, cap).pin_memory() for n in ("q", "k", "v", "do")}
    sh = {n: t.to(dev) for n, t in host.items()}
    # device buffers of the step (allocated once; the step itself allocates nothing)
    yq, yk, yv, ydo = (torch.empty((P, B, S, Hg, D), dtype=torch.bfloat16, device=dev) for _ in range(4))
    yo, ydq, ydk, ydv = (torch.empty_like(yq) for _ in range(4))
    lse = torch.empty((P, B, Hg, S), dtype=torch.float32, device=dev)
    o_sh, dq_sh, dk_sh, dv_sh = (torch.empty_like(sh["q"]) for _ in range(4))
    fused_bwd = args.bwd == "fused"
    ws_bytes = (uaa.attn_bwd_fused_workspace_bytes if fused_bwd else uaa.attn_bwd_workspace_bytes)(P * B, S, Hg, D)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    fused = args.path == "fused"
    if fused:
        # the exchanges fused into the attention kernels: the step reads and writes the shards only
        lse_f = torch.empty((B, H, S), dtype=torch.float32, device=dev)
        ws = torch.empty(uaa.ulysses_attn_bwd_workspace_bytes(lens, cap, B, H, D), dtype=torch.uint8, device=dev)
        del yq, yk, yv, ydo, yo, ydq, ydk, ydv, lse
    stream = torch.cuda.current_stream(dev)
    ev = {}
    # per-call events around the backward's dK/dV and dQ kernels (created and recorded once up front)
    prof = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for trio in prof:
        for e in trio:
            e.record(stream)
    prof_iter = iter(prof)

    def mark(name):
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        ev.setdefault(name, []).append(e)

    def step_fused(timed=False, bufs=None):
        src = bufs or sh
        if timed:
            mark("fwd0")
        uaa.ulysses_attn_fwd(src["q"], src["k"], src["v"], lens, None, w.scale, out=o_sh, lse=lse_f)
        if timed:
            mark("fwd1")
            mark("bwd0")
            uaa.set_bwd_profile_events(next(prof_iter))
        uaa.ulysses_attn_bwd(src["q"], src["k"], src["v"], o_sh, src["do"], lse_f, lens, None, w.scale, dq=dq_sh,
                             dk=dk_sh, dv=dv_sh, workspace=ws)
        if timed:
            uaa.set_bwd_profile_events(None)
            mark("bwd1")

    def step(timed=False):
        if fused:
            return step_fused(timed)
        if timed:
            mark("s2h_fwd0")
        for n, y in (("q", yq), ("k", yk), ("v", yv)):
            uaa.seq_to_head(sh[n], lens, out=y)
        if timed:
            mark("s2h_fwd1")
        if timed:
            mark("fwd0")
        # all P head groups in one launch: (P, B, N, Hg, D) is a BSHD tensor of batch P*B
        uaa.attn_fwd(yq.view(P * B, S, Hg, D), yk.view(P * B, S, Hg, D), yv.view(P * B, S, Hg, D), None, w.scale,
                     out=yo.view(P * B, S, Hg, D), lse=lse.view(P * B, Hg, S))
        if timed:
            mark("fwd1")
        if timed:
            mark("h2s_o0")
        uaa.head_to_seq(yo, lens, cap, out=o_sh)
        uaa.seq_to_head(sh["do"], lens, out=ydo)
        if timed:
            mark("h2s_o1")
        if timed:
            mark("bwd0")
            uaa.set_bwd_profile_events(next(prof_iter))
        g4 = lambda t: t.view(P * B, S, Hg, D)  # noqa: E731
        uaa.attn_bwd(g4(yq), g4(yk), g4(yv), g4(yo), g4(ydo), lse.view(P * B, Hg, S), None, w.scale, dq=g4(ydq),
                     dk=g4(ydk), dv=g4(ydv), workspace=ws, fused=fused_bwd)
        if timed:
            uaa.set_bwd_profile_events(None)
            mark("bwd1")
        if timed:
            mark("h2s_g0")
        for y, x in ((ydq, dq_sh), (ydk, dk_sh), (ydv, dv_sh)):
            uaa.head_to_seq(y, lens, cap, out=x)
        if timed:
            mark("h2s_g1")

    # exchange path: 3 seq->head, forward, head->seq (O), seq->head (dO), preprocess + dK/dV + dQ,
    # 3 head->seq; fused path: padding fill + forward, 3 padding fills + preprocess + dK/dV + dQ
    launches_per_step = (2 + 6) if fused else (3 + 1 + 1 + 1 + 3 + 3)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    uaa.check_device_status(dev)

    barrier(world)
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for _ in range(args.steps):
            step(timed=True)
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    uaa.check_device_status(dev)
    ms = t_start.elapsed_time(t_end) / args.steps
    ms = max_over_ranks(world, ms)

    def pair_ms(a, b):
        return sum(x.elapsed_time(y) for x, y in zip(ev[a], ev[b]))

    if fused:
        for k in ("s2h_fwd0", "s2h_fwd1", "h2s_o0", "h2s_o1", "h2s_g0", "h2s_g1"):
            ev[k] = []
    fwd_ms = pair_ms("fwd0", "fwd1") / args.steps
    bwd_ms = pair_ms("bwd0", "bwd1") / args.steps
    fwd_launch = pair_ms("fwd0", "fwd1") / len(ev["fwd0"])
    bwd_launch = pair_ms("bwd0", "bwd1") / len(ev["bwd0"])
    relayout_ms = (pair_ms("s2h_fwd0", "s2h_fwd1") + pair_ms("h2s_o0", "h2s_o1") +
                   pair_ms("h2s_g0", "h2s_g1")) / args.steps
    tensor_bytes = B * S * H * D * 2
    relayout_bytes = 8 * 2 * tensor_bytes + 4 * (P * B * cap * H * D * 2 - tensor_bytes)  # + padding zero fill
    if fused:
        relayout_bytes = 0
    step_flops = flops(B, S, H, D)
    value = world * step_flops / (ms * 1e-3) / 1e12

    # e2e through the same public calls with host buffers: every step copies its input shards (Q, K,
    # V, dO) from pinned host memory and reads O, dQ, dK, dV back, inside the timed region.  The copies
    # run on two copy streams ordered against the compute stream by events: dO arrives while the
    # forward runs, O leaves while the backward runs, and the next step's Q, K, V arrive as soon as
    # this step's seq->head exchange has consumed the previous ones (device buffers are reused).
    outs_host = {n: torch.empty_like(host["q"]).pin_memory() for n in ("o", "dq", "dk", "dv")}
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    e_qkv_in, e_do_in, e_qkv_free, e_do_free, e_o_ready, e_g_ready, e_o_out, e_g_out = (
        torch.cuda.Event() for _ in range(8))
    for e in (e_qkv_free, e_do_free, e_o_out, e_g_out):
        e.record(stream)

    def e2e_step():
        with torch.cuda.stream(h2d_s):
            h2d_s.wait_event(e_qkv_free)
            for n in ("q", "k", "v"):
                sh[n].copy_(host[n], non_blocking=True)
            e_qkv_in.record(h2d_s)
            h2d_s.wait_event(e_do_free)
            sh["do"].copy_(host["do"], non_blocking=True)
            e_do_in.record(h2d_s)
        stream.wait_event(e_qkv_in)
        for n, y in (("q", yq), ("k", yk), ("v", yv)):
            uaa.seq_to_head(sh[n], lens, out=y)
        e_qkv_free.record(stream)
        uaa.attn_fwd(yq.view(P * B, S, Hg, D), yk.view(P * B, S, Hg, D), yv.view(P * B, S, Hg, D), None, w.scale,
                     out=yo.view(P * B, S, Hg, D), lse=lse.view(P * B, Hg, S))
        stream.wait_event(e_o_out)  # the previous step's read-back of O is done with o_sh
        uaa.head_to_seq(yo, lens, cap, out=o_sh)
        e_o_ready.record(stream)
        stream.wait_event(e_do_in)
        uaa.seq_to_head(sh["do"], lens, out=ydo)
        e_do_free.record(stream)
        g4 = lambda t: t.view(P * B, S, Hg, D)  # noqa: E731
        uaa.attn_bwd(g4(yq), g4(yk), g4(yv), g4(yo), g4(ydo), lse.view(P * B, Hg, S), None, w.scale, dq=g4(ydq),
                     dk=g4(ydk), dv=g4(ydv), workspace=ws, fused=fused_bwd)
        stream.wait_event(e_g_out)  # the previous step's read-back of the gradients is done
        for y, x in ((ydq, dq_sh), (ydk, dk_sh), (ydv, dv_sh)):
            uaa.head_to_seq(y, lens, cap, out=x)
        e_g_ready.record(stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(e_o_ready)
            outs_host["o"].copy_(o_sh, non_blocking=True)
            e_o_out.record(d2h_s)
            d2h_s.wait_event(e_g_ready)
            for n, t in (("dq", dq_sh), ("dk", dk_sh), ("dv", dv_sh)):
                outs_host[n].copy_(t, non_blocking=True)
            e_g_out.record(d2h_s)

    # fused path: the backward reads the input shards again, so two input buffer sets alternate and
    # the next step's inputs arrive while this step computes
    sh2 = {n: torch.empty_like(t) for n, t in sh.items()} if fused and not args.no_e2e else None
    e_in_free = [torch.cuda.Event(), torch.cuda.Event()]
    e_in_ready = [torch.cuda.Event(), torch.cuda.Event()]
    for e in e_in_free:
        e.record(stream)
    e2e_i = [0]

    def e2e_step_fused():
        i = e2e_i[0] % 2
        e2e_i[0] += 1
        bufs = sh if i == 0 else sh2
        with torch.cuda.stream(h2d_s):
            h2d_s.wait_event(e_in_free[i])
            for n in ("q", "k", "v", "do"):
                bufs[n].copy_(host[n], non_blocking=True)
            e_in_ready[i].record(h2d_s)
        stream.wait_event(e_in_ready[i])
        stream.wait_event(e_o_out)  # the previous step's read-back of O is done with o_sh
        uaa.ulysses_attn_fwd(bufs["q"], bufs["k"], bufs["v"], lens, None, w.scale, out=o_sh, lse=lse_f)
        e_o_ready.record(stream)
        stream.wait_event(e_g_out)  # the previous step's read-back of the gradients is done
        uaa.ulysses_attn_bwd(bufs["q"], bufs["k"], bufs["v"], o_sh, bufs["do"], lse_f, lens, None, w.scale,
                             dq=dq_sh, dk=dk_sh, dv=dv_sh, workspace=ws)
        e_in_free[i].record(stream)
        e_g_ready.record(stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(e_o_ready)
            outs_host["o"].copy_(o_sh, non_blocking=True)
            e_o_out.record(d2h_s)
            d2h_s.wait_event(e_g_ready)
            for n, t in (("dq", dq_sh), ("dk", dk_sh), ("dv", dv_sh)):
                outs_host[n].copy_(t, non_blocking=True)
            e_g_out.record(d2h_s)

    if fused:
        e2e_step = e2e_step_fused  # noqa: F811

    def host_link():
        """One step's copies alone (no compute), H2D and D2H concurrently on the two copy
        streams: the floor the e2e step cannot go below, whatever the overlap."""
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        h2d_s.wait_event(a)
        d2h_s.wait_event(a)
        with torch.cuda.stream(h2d_s):
            for n in ("q", "k", "v", "do"):
                sh[n].copy_(host[n], non_blocking=True)
        with torch.cuda.stream(d2h_s):
            for n, t in (("o", o_sh), ("dq", dq_sh), ("dk", dk_sh), ("dv", dv_sh)):
                outs_host[n].copy_(t, non_blocking=True)
        stream.wait_stream(h2d_s)
        stream.wait_stream(d2h_s)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    e2e = None
    if not args.no_e2e:
        link_ms = min(host_link() for _ in range(3))
        e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with Clocks(local) as clk_e2e:  # this loop follows the device-timed one on a warm GPU
            e0.record(stream)
            h2d_s.wait_event(e0)
            d2h_s.wait_event(e0)
            for _ in range(args.steps):
                e2e_step()
            stream.wait_stream(h2d_s)
            stream.wait_stream(d2h_s)
            e1.record(stream)
            torch.cuda.synchronize()
        e2e_ms = max_over_ranks(world, e0.elapsed_time(e1) / args.steps)
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = sum(t.numel() * t.element_size() for t in outs_host.values())
        e2e = {"value": world * step_flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "copies": "two copy streams overlapped with compute (event-ordered)",
               "copies_alone_ms_per_step": link_ms,
               "host_link_gbs": (h2d + d2h) / (link_ms * 1e-3) / 1e9,
               "clocks": clk_e2e.summary()}
    uaa.check_device_status(dev)

    pk, src = peaks()
    peak_tf, key = _peak_value(pk, "bf16_tflops_sustained", "bf16_tflops")
    peak_hbm, _ = _peak_value(pk, "hbm_gbs")
    dkdv_ms = sum(a.elapsed_time(b) for a, b, _ in prof) / len(prof)
    dq_ms = sum(b.elapsed_time(c) for _, b, c in prof) / len(prof)
    # dominant kernel: the split dK/dV kernel (S, dP, dV, dK GEMMs of all P head groups = 8*P*B*Hg*S^2*D
    # algorithmic FLOPs) or the one-pass backward kernel (the same plus dQ: 10*P*B*Hg*S^2*D)
    dkdv_flops = (10 if fused_bwd else 8) * P * B * Hg * S * S * D
    achieved = dkdv_flops / (dkdv_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                "frac": achieved / peak_tf, "traffic": None if fused_bwd else dkdv_traffic(),
                "kernel": ("attn_bwd_fused_kernel<128,false> (all head groups: S, dP, dV, dK, dQ GEMMs)" if fused_bwd
                           else "attn_bwd_dkdv_kernel<128,false> (all head groups: S, dP, dV, dK GEMMs)"),
                "flops_per_launch": dkdv_flops, "ms_per_launch": dkdv_ms,
                "peak_source": f"{src} {key}"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        f, t, desc = oracle_sample(inp, w, seconds=args.cpu_seconds)
        cpu = {"value": f / t / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle", "sample": desc}
    line = {
        "metric": "attention fwd+bwd TFLOP/s", "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_name, "B": B, "N": S, "P": P, "H": H, "D": D, "shard_lens": list(lens),
                   "cap": cap, "mask": None, "l2": "inputs larger than L2 (4 x 279 MB shards), no flush",
                   "path": "exchanges fused into the attention kernels" if fused else
                   "seq->head / head->seq re-layout kernels around the attention kernels",
                   "bwd": "one pass, dQ by fp32 reductions" if fused_bwd else "split dK/dV and dQ passes",
                   "parallelism": "replicas" if world > 1 else "single GPU, 4 emulated Ulysses ranks"},
        "parts_ms_per_step": {"attn_fwd": fwd_ms, "attn_bwd": bwd_ms, "relayout": relayout_ms},
        "attn_fwd_tflops": flops(B, S, H, D, bwd=False) / (fwd_ms * 1e-3) / 1e12,
        "attn_bwd_tflops": flops(B, S, H, D, fwd=False) / (bwd_ms * 1e-3) / 1e12,
        "fwd_launch_tflops": flops(P * B, S, Hg, D, bwd=False) / (fwd_launch * 1e-3) / 1e12,
        "kernel_ms_per_launch": ({"attn_fwd_kernel": fwd_launch, "attn_bwd_fused_kernel": dkdv_ms,
                                  "dq_convert_kernel": dq_ms} if fused_bwd else
                                 {"attn_fwd_kernel": fwd_launch, "attn_bwd_dkdv_kernel": dkdv_ms,
                                  "attn_bwd_dq_kernel": dq_ms}),
        "dq_kernel_tflops": None if fused_bwd else (6 * P * B * Hg * S * S * D) / (dq_ms * 1e-3) / 1e12,
        "relayout_gbs": relayout_bytes / (relayout_ms * 1e-3) / 1e9 if relayout_ms > 0 else None,
        "relayout_hbm_frac": ((relayout_bytes / (relayout_ms * 1e-3) / 1e9) / peak_hbm
                              if peak_hbm and relayout_ms > 0 else None),
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not args.no_configs and not args.heads:
        # the other workloads, each timed on its own after the headline (not part of its step)
        line["per_config"] = run_configs(uaa, args, dev, local)
    if rank == 0:
        print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="uaa", choices=["uaa", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload records of the layout, 1k DiT, masked and full-layer workloads")
    ap.add_argument("--cpu-config-seconds", type=float, default=30.0,
                    help="host-time budget of the oracle per workload record (0: skip)")
    ap.add_argument("--heads", type=int, default=0, help="override H (profiling-size variant)")
    ap.add_argument("--bwd", default="split", choices=["split", "fused"],
                    help="backward: split dK/dV + dQ passes (bit-reproducible) or one pass with dQ reductions")
    ap.add_argument("--workload", default=None, choices=[w.name for w in synth.WORKLOADS],
                    help="time only this workload's fwd / bwd / fwd+bwd record (no headline line)")
    ap.add_argument("--path", default="exchange", choices=["fused", "exchange"],
                    help="Ulysses step: attention kernels reading the shards directly, or separate re-layouts")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "uaa" else args.warmup
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        run_reference(args, world, rank)
        return
    world, rank, local = dist_setup(args.gpus)
    if args.workload:
        run_one_workload(args, local)
    else:
        run_gpu(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
