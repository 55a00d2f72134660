"""Benchmark of the chunked gated delta rule forward on GB300.

One step = the whole forward of one batch of the workload: q/k prep, the
intra-chunk WY kernel and the chunk-serial state/output kernel (both scan
directions and the denominator for the bidirectional workload), on inputs
already resident in HBM. Default workload: causal, bf16 q/k/v with fp32
state and gates, B=4, H=16, T=4096, K=V=128, chunk 64 (inputs ~275 MB, larger
than the 129 MB L2, so no flush is needed between steps).

Prints one JSON line (rank 0). `--impl reference` times the fp64 CPU oracle
(the reference arm) on a bounded sample of the same workload instead.
Multi-GPU (torchrun, one rank per GPU): every rank runs its own replica of the
workload with its own seed (weak scaling, no collective on the data path);
the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "GDN chunked fwd tokens/s & TFLOP/s at 1 GB300; % of roofline; vs CPU oracle"
DEFAULT_WORKLOAD = "causal_bf16_b4h16t4096d128"
C = 64
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Nominal FP32 FFMA peak of the part (MEASURED_PEAKS.json has no fp32 figure):
# 152 SMs x 128 FP32 lanes x 2 FLOP x 2.07 GHz maximum SM clock.
FP32_TFLOPS_NOMINAL = 152 * 128 * 2 * 2.07e9 / 1e12
# L2 size used to decide whether inputs fit in L2 (then the timed steps are
# each preceded by an L2 flush): 129 MB, the same number in both arms.
L2_BYTES = 129 * 10 ** 6
# The five workloads of the benchmark statement, reported side by side.
CONFIGS = ["causal_f32_b1h2t256d64", "causal_bf16_b4h16t4096d128", "bidir_video_b2h16n8192d112",
           "varlen_bf16_64seq_h32d128", "gk_bf16_b1h32t65536k128v256"]
# the timed steps plus this much more of the same step, back to back, are
# sampled for clocks (nvidia-smi needs a run of about a second to see it)
CLOCK_SOAK_S = 1.5


# ------------------------------------------------------------ work model ---

def flops_per_token_head(K, V, C=C):
    """Algorithmic FLOPs per (token, head) of one scan direction: w h, the
    state update and q h (2KV each), strictly lower K K^T, T X and T Y (half
    triangles), the intra-chunk output pair, and the forward substitution
    (C^3/3 per chunk)."""
    return 6.0 * K * V + 3.0 * C * K + 2.0 * C * V + C * C / 3.0


def path_work(w):
    """(algorithmic FLOPs, minimum HBM bytes) of one step of workload w:
    inputs read once, outputs written once, h0/h_final once."""
    th = w.B * w.T * w.H
    e = 2 if w.dtype == "bf16" else 4
    if w.frame > 1:
        # per token-head: the frame Gram K^T diag(beta)[K | V | 1] and O = Q S (2KVt
        # each direction summed first); the chain adds 2 K K Vt per frame and direction
        Vt = w.V + (1 if w.bidirectional else 0)
        dirs = 2 if w.bidirectional else 1
        fl = th * (2.0 * w.K * (w.K + Vt) + 2.0 * w.K * Vt) + dirs * w.B * w.H * (w.T // w.frame) \
            * 2.0 * w.K * w.K * Vt
        by = th * (3 * w.K * e + 4 + w.V * e + (4 if w.bidirectional else 0)) \
            + w.B * w.H * (w.T // w.frame) * 4
        if w.h0 is not None:
            by += w.n_seq * w.H * w.K * w.V * 4
        if not w.bidirectional:
            by += w.n_seq * w.H * w.K * w.V * 4
        return fl, by
    if w.bidirectional:
        fl = th * (flops_per_token_head(w.K, w.V) + flops_per_token_head(w.K, w.V + 1))
        by = th * (3 * w.K * e + 4 + 4 + w.V * e + 4)       # qkv, beta, g, num, den
        if w.g_bwd is not None or w.beta_bwd is not None:
            by += th * 8                                     # backward gates and beta
        if w.merge:
            fl += th * w.V * (6 if w.gate is not None else 2)
            by += th * w.V * e * (2 if w.gate is not None else 1)  # gate in, merged out
    else:
        fl = th * flops_per_token_head(w.K, w.V)
        by = th * ((2 * w.K + w.V) * e + 4 + (4 * w.K if w.gk is not None else 4) + w.V * e)
        if w.h0 is not None:
            by += w.n_seq * w.H * w.K * w.V * 4
        by += w.n_seq * w.H * w.K * w.V * 4                 # h_final
    return fl, by


METRIC_BWD = "GDN chunked bwd tokens/s (forward recompute + all input gradients) at 1 GB300"


def seg_count(w):
    """Segments per sequence of a segment-parallel workload (1 otherwise)."""
    if not isinstance(w.segment_len, int) or w.segment_len <= 0:
        return 1
    return -(-(-(-w.T // C)) // (w.segment_len // C))


def kernel_bytes(w, name):
    """Algorithmic bytes one launch of kernel `name` must move for workload
    w: its own inputs read once and outputs written once (shared tiles counted
    once, padding not counted)."""
    th = w.B * w.T * w.H
    e = 2 if w.dtype == "bf16" else 4
    K, V = w.K, w.V + (1 if w.bidirectional else 0)
    gate = 4 * w.K if w.gk is not None else 4
    chunks = th / C
    if name == "intra_bf16":
        return th * ((2 * K + w.V) * e + 4 + gate + (3 * K + V + C) * 2) + chunks * K * 4
    if name == "fused_tc":  # one direction: q, k, v, beta, g in; o (and den) out; h0 / h_final
        hs = 0 if w.bidirectional else (2 if w.h0 is not None else 1) * w.n_seq * w.H * w.K * w.V * 4
        return th * ((2 * w.K + w.V) * e + 8 + w.V * e + (4 if w.bidirectional else 0)) + hs
    n_seg, bh = seg_count(w), w.n_seq * w.H
    if name == "state_tc":
        hs = (2 if w.h0 is not None else 1) * w.n_seq * w.H * w.K * w.V * 4
        if n_seg > 1:  # each segment reads the state entering it
            hs += (n_seg - (1 if w.h0 is not None else 0)) * bh * K * V * 4
        return th * ((3 * K + V + C) * 2 + w.V * e + (4 if w.bidirectional else 0)) \
            + chunks * K * 4 + (0 if w.bidirectional else hs)
    if name == "seg_summary":  # every segment but the last: images in, (E, M) out
        f = (n_seg - 1) / n_seg
        return f * (th * ((3 * K + V + C) * 2) + chunks * K * 4) + (n_seg - 1) * bh * K * (V + K) * 4
    if name == "seg_combine":  # (E, M) in, the entering states out
        return (n_seg - 1) * bh * K * (V + K) * 4 + n_seg * bh * K * V * 4
    if name == "f32_prep":  # inputs in; w, qg, kg, P, u images and dec out (fp32)
        return th * ((2 * K + w.V) * e + 4 + gate + (3 * K + C + V) * 4) + chunks * K * 4
    if name == "f32_serial":  # the images in, the output (and h0 / h_final) out
        return th * ((3 * K + C + V) * 4 + w.V * e) + chunks * K * 4 + \
            (2 if w.h0 is not None else 1) * w.n_seq * w.H * w.K * w.V * 4
    if name == "fused_f32":
        return th * ((2 * K + w.V) * e + 4 + gate + w.V * e) + w.n_seq * w.H * w.K * w.V * 4
    if name == "prep_rms":
        return w.B * w.T * w.H * w.K * e * 2 + w.B * w.T * 4
    if name == "prep_l2":
        return th * w.K * e * 2
    if name in ("frame_gram", "frame_chain", "frame_out"):
        Vt = w.V + (1 if w.bidirectional else 0)
        nf = w.B * w.H * (w.T // w.frame)
        mats = nf * w.K * (w.K + Vt) * 4          # A_f and B_f, fp32
        states = nf * w.K * Vt * 4                 # the states the outputs read
        if name == "frame_gram":                   # k, v, beta in; A_f, B_f out
            return th * (w.K * e + w.V * e + 4) + mats
        if name == "frame_chain":                  # A_f, B_f in; states out
            return mats + states + nf * 4
        return th * (w.K * e + w.V * e + (4 if w.bidirectional else 0)) + states
    if name == "merge":
        return th * w.V * e * (3 if w.gate is not None else 2) + th * 4
    snap_h = w.B * w.H * (-(-w.T // C)) * w.K * w.V * 2  # one bf16 K x V state per chunk
    snap_v = th * w.V * 2                                 # one bf16 value row per token
    if name == "bwd_dh":  # images + do in; dh' and dv_new snapshots out
        return th * ((3 * K + C) * 2 + w.V * 2) + chunks * K * 4 + snap_h + snap_v
    if name == "bwd_dq":  # q, k, do, v_new, h in; dq, dk and dG partials out
        return th * (2 * K * 2 + w.V * 2 + 4) + snap_v + snap_h + th * (2 * K * 4 + 4)
    if name == "bwd_dk":  # k, v, dv_new, v_new, h, dh', partials in; dk, dv, dbeta, dg out
        return th * (K * 2 + w.V * 2 + 8) + 2 * snap_v + 2 * snap_h + th * (K * 4 + 4) \
            + th * (K * 4 + w.V * 4 + 8)
    return None


KERNEL_SOURCES = {"fused_tc": ["gdn_fused_tc.cu", "gdn_tc.cuh", "gdn_common.cuh"],
                  "intra_bf16": ["gdn_intra_bf16.cu", "gdn_common.cuh"],
                  "state_tc": ["gdn_state_tc.cu", "gdn_tc.cuh", "gdn_common.cuh"]}


def measured_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, or None when no
    capture exists for this kernel and workload or the kernel's sources have
    changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if kernel not in KERNEL_SOURCES or not os.path.exists(path):
        return None
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "gated_delta_rule_18_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    digest = h.hexdigest()[:16]
    with open(path) as fh:
        for line in fh:
            parts = line.split()
            if len(parts) == 4 and not line.startswith("#") and parts[0] == kernel \
                    and parts[1] == workload and parts[3] == digest:
                return int(parts[2])
    return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------- multi-rank ----

def max_over_ranks(x, dist=None, device=None):
    """The largest value of x over all ranks (the job takes as long as its
    slowest replica); identity without a process group."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank, world, steps, seconds):
    """Whole-job throughput: every rank processed its own replica of the
    workload (weak scaling), so the job processed world x tokens per step."""
    return tokens_per_rank * world * steps / seconds


# --------------------------------------------------------------- clocks ----

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ----------------------------------------------------------- device side ---

def device_inputs(w, dev):
    import torch

    def to_dev(st):
        if st.dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(st.bits).view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(st.values)).to(dev)

    def f32(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)

    d = {}
    if w.qkv is not None:
        qkv = to_dev(w.qkv)
        d["qkv"] = qkv
        d["q"], d["k"], d["v"] = qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2]
    else:
        d["q"], d["k"], d["v"] = to_dev(w.q), to_dev(w.k), to_dev(w.v)
    d["beta"], d["g"], d["gk"], d["h0"] = f32(w.beta), f32(w.g), f32(w.gk), f32(w.h0)
    d["g_bwd"], d["beta_bwd"] = f32(w.g_bwd), f32(w.beta_bwd)
    d["g_frame"] = f32(w.g_frame)
    d["gate"] = None if w.gate is None else to_dev(w.gate)
    d["cu_seqlens"] = None if w.cu_seqlens is None else torch.from_numpy(
        w.cu_seqlens.astype(np.int32)).to(dev)
    return d


def run_step(gdn, w, d, ws):
    extra = {}
    if w.segment_len is not None:
        extra["segment_len"] = w.segment_len
    if w.frame > 1:
        extra = dict(frame=w.frame, g_frame=d["g_frame"])
    elif w.bidirectional:
        bw = {k2: d[k2 + "_bwd"] for k2 in ("g", "beta") if d.get(k2 + "_bwd") is not None}
        extra = dict(backward=bw or None, merge=w.merge, gate=d.get("gate"), eps=w.eps)
    return gdn.gdn_forward(d["q"], d["k"], d["v"], d["beta"], g=d["g"], gk=d["gk"],
                           h0=d["h0"], cu_seqlens=d["cu_seqlens"], prep=w.prep,
                           bidirectional=w.bidirectional,
                           with_final_state=not w.bidirectional, workspace=ws, **extra)


def resolve_segments(gdn, w, dev):
    """The workload with its segment length fixed for this device (the
    library's choice for "auto")."""
    import torch
    if w.segment_len != "auto":
        return w
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    return dataclasses.replace(w, segment_len=gdn.gdn_seg_choose(
        w.B, w.T, w.H, w.K, w.V, w.bidirectional, n_sm))


def workspace_for(gdn, w, dev):
    import torch
    dt = gdn.BF16 if w.dtype == "bf16" else gdn.F32
    if w.segment_len is not None:
        n = gdn.gdn_seg_workspace_size(w.B, w.T, w.H, w.K, w.V, w.bidirectional, w.segment_len)
        return torch.empty(max(n, 256), dtype=torch.uint8, device=dev)
    if w.bidirectional and w.frame == 1:  # both directions at once (two workspaces + staging)
        n = gdn.gdn_bidir_workspace_size(w.B, w.T, w.H, w.K, w.V, w.n_seq, w.cu_seqlens is not None,
                                         dt, True)
        return torch.empty(max(n, 256), dtype=torch.uint8, device=dev)
    n = gdn.gdn_workspace_size(w.B, w.T, w.H, w.K, w.V, w.n_seq, w.cu_seqlens is not None, dt,
                               w.bidirectional)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=dev)


def e2e_measure(gdn, w, d, ws, steps, dev):
    """The same forward through the public API with pinned host buffers:
    every step copies its inputs host->device, runs, and copies its output
    back. Steps are pipelined the way a serving loop would run them: two
    sets of device input buffers, the copies in on one stream and out on
    another, so that step i+1's inputs arrive while step i computes and step
    i-1's output leaves. The timed region spans the first copy in to the last
    copy out."""
    import torch
    host = {}
    for key in ("qkv", "q", "k", "v", "beta", "g", "gk", "h0", "cu_seqlens", "g_bwd",
                "beta_bwd", "gate", "g_frame"):
        t = d.get(key)
        if t is None or (key in ("q", "k", "v") and "qkv" in d):
            continue
        host[key] = t.detach().to("cpu").contiguous().pin_memory() if t.is_contiguous() else None
    if "qkv" not in d:
        for key in ("q", "k", "v"):
            host[key] = d[key].to("cpu").pin_memory()
    bufs = [{k2: torch.empty_like(v2, device=dev) for k2, v2 in host.items() if v2 is not None}
            for _ in range(2)]
    out_shape = (w.B, w.T, w.H, w.V)
    out_host = torch.empty(out_shape, dtype=d["v"].dtype).pin_memory()
    h2d = sum(v2.numel() * v2.element_size() for v2 in host.values() if v2 is not None)
    d2h = out_host.numel() * out_host.element_size()
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    in_done = [torch.cuda.Event() for _ in range(2)]
    used = [torch.cuda.Event() for _ in range(2)]  # step on buffer b has read its inputs
    for e in used:
        e.record(comp)

    def one(i):
        bb = bufs[i % 2]
        s_in.wait_event(used[i % 2])
        with torch.cuda.stream(s_in):
            for k2, v2 in host.items():
                if v2 is not None:
                    bb[k2].copy_(v2, non_blocking=True)
        in_done[i % 2].record(s_in)
        comp.wait_event(in_done[i % 2])
        dd = dict(d)
        dd.update(bb)
        if "qkv" in bb:
            qkv = bb["qkv"]
            dd["q"], dd["k"], dd["v"] = qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2]
        res = run_step(gdn, w, dd, ws)
        used[i % 2].record(comp)
        o = res["merged" if w.merge else "out"]
        o.record_stream(s_out)
        s_out.wait_event(used[i % 2])
        with torch.cuda.stream(s_out):
            out_host.copy_(o, non_blocking=True)

    for i in range(2):
        one(i)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(comp)
    s_in.wait_event(a)
    for i in range(steps):
        one(i)
    done = torch.cuda.Event()
    done.record(s_out)
    comp.wait_event(done)
    b.record(comp)
    b.synchronize()
    sec = a.elapsed_time(b) / 1e3 / steps
    return sec, h2d, d2h


PROFILE_EVERY = 4


def graph_replay(gdn, w, d, ws, n, fl, by, peaks, reps=20):
    """N back-to-back calls of the step captured in one CUDA graph and
    replayed: the per-call time with the launch cost amortised (the CPU
    enqueues nothing per call). The library's per-launch event pairs are off
    here (they are on only in the timed region above)."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            run_step(gdn, w, d, ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(n):
            run_step(gdn, w, d, ws)
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    per_call = a.elapsed_time(b) / 1e3 / (reps * n)
    roof = max(by / (peaks["hbm_gbs"] * 1e9), fl / (peaks["bf16_tflops"] * 1e12))
    return {"calls_per_graph": n, "replays": reps, "us_per_call": per_call * 1e6,
            "l2": "warm: no flush between the calls of a replay",
            "tokens_per_s": w.B * w.T / per_call if w.cu_seqlens is None else int(w.cu_seqlens[-1]) / per_call,
            "path_roofline_frac": roof / per_call}


# ------------------------------------------------------------- CPU side ----

ORACLE_S_PER_TOKEN_HEAD_KV = 7e-9   # rough fp64 oracle cost per token-head per K*V
CPU_TARGET_CORE_SECONDS = 40.0


def oracle_sample(w):
    """Time the fp64 oracle (as it stands, all host cores) on a bounded sample
    of workload w: leading batch rows / sequences and heads, sized to about
    CPU_TARGET_CORE_SECONDS of single-core work. Returns (tokens/s of the full
    workload equivalent, seconds, threads used, description)."""
    import dataclasses

    import oracle
    threads = os.cpu_count() or 1
    target = CPU_TARGET_CORE_SECONDS / (ORACLE_S_PER_TOKEN_HEAD_KV * w.K * w.V)
    if w.qkv is not None:
        # full-channel RMS prep needs every head of a token: whole batch rows
        ix = (slice(0, 1),)
        sw = dataclasses.replace(w, B=1, qkv=w.qkv.take(ix), q=w.q.take(ix), k=w.k.take(ix),
                                 v=w.v.take(ix), beta=w.beta[ix],
                                 g=None if w.g is None else w.g[ix],
                                 g_frame=None if w.g_frame is None else w.g_frame[ix],
                                 g_bwd=None if w.g_bwd is None else w.g_bwd[ix],
                                 beta_bwd=None if w.beta_bwd is None else w.beta_bwd[ix],
                                 gate=None if w.gate is None else w.gate.take(ix))
        desc = (f"batch row 0 of {w.B}: {w.T} tokens x {w.H} heads, both directions + den"
                + (" + merge" if w.merge else ""))
        units = w.H
    elif w.cu_seqlens is not None:
        cu = w.cu_seqlens
        nh = w.H
        ns = 1
        while ns < w.n_seq and cu[ns] * nh < target:
            ns += 1
        if cu[ns] * nh > 2 * target:
            nh = max(1, int(target // max(1, cu[ns])))
        ix = (slice(None), slice(0, int(cu[ns])), slice(0, nh))
        sw = dataclasses.replace(w, T=int(cu[ns]), H=nh, q=w.q.take(ix), k=w.k.take(ix),
                                 v=w.v.take(ix), beta=w.beta[ix], g=w.g[ix],
                                 h0=w.h0[:ns, :nh], cu_seqlens=cu[:ns + 1])
        desc = f"sequences 0..{ns - 1} ({int(cu[ns])} tokens) x heads 0..{nh - 1} of {w.H}"
        units = ns * nh
    else:
        n_units = int(max(1, min(w.B * w.H, round(target / max(1, w.T)))))
        nb = min(w.B, -(-n_units // w.H))
        nh = w.H if nb > 1 else n_units
        ix = (slice(0, nb), slice(None), slice(0, nh))
        sw = dataclasses.replace(w, B=nb, H=nh, q=w.q.take(ix), k=w.k.take(ix),
                                 v=w.v.take(ix), beta=w.beta[ix],
                                 g=None if w.g is None else w.g[ix],
                                 gk=None if w.gk is None else w.gk[ix],
                                 h0=None if w.h0 is None else w.h0[:nb, :nh])
        desc = f"batch rows 0..{nb - 1} of {w.B} x heads 0..{nh - 1} of {w.H}, {w.T} tokens"
        units = nb * nh
    t0 = time.perf_counter()
    oracle.forward(sw, threads=threads)
    sec = time.perf_counter() - t0
    token_heads = sw.B * sw.T * sw.H
    return token_heads / w.H / sec, sec, min(threads, units), desc


# ------------------------------------------------------------------ main ---

def workload_input_bytes(w):
    """Bytes of the workload's input tensors as they sit in HBM (qkv counted
    once when q, k, v are views of it)."""
    n = 0
    for st in ((w.qkv,) if w.qkv is not None else (w.q, w.k, w.v)):
        n += int(np.prod(st.shape)) * (2 if st.dtype == "bf16" else 4)
    for a in (w.beta, w.g, w.gk, w.h0, w.g_bwd, w.beta_bwd, w.g_frame, w.cu_seqlens):
        if a is not None:
            n += int(np.asarray(a).size) * 4
    if w.gate is not None:
        n += int(np.prod(w.gate.shape)) * 2
    return n


def workload_tokens(w):
    return w.B * w.T


def config_of(w, name, world):
    """The `config` object of the JSON line (the same in both arms) and
    whether the timed steps are preceded by an L2 flush (inputs that fit in
    L2)."""
    in_bytes = workload_input_bytes(w)
    flush = in_bytes <= L2_BYTES
    cfg = {"workload": name, "B": w.B, "T": w.T, "H": w.H, "K": w.K, "V": w.V, "chunk": C,
           "tokens_per_step_per_gpu": workload_tokens(w),
           "l2": ("L2 flushed before every timed step (2 x L2 bytes written, outside the "
                  "step's events)" if flush else "inputs larger than L2 (no flush)"),
           "input_bytes": in_bytes, "parallelism": f"replicas x{world}"}
    if w.segment_len is not None:
        cfg.update(segment_len=w.segment_len, segments=seg_count(w))
    return cfg, flush


def path_roof(w, peaks):
    """(FLOPs, bytes, roofline seconds, bound, compute peak TFLOP/s, its
    source) of one step of w: bf16 workloads against the measured dense bf16
    tensor peak, fp32 ones against the nominal FP32 FFMA peak."""
    fl, by = path_work(w)
    if w.dtype == "bf16":
        pk, src = peaks["bf16_tflops"], "bf16_tflops"
    else:
        pk, src = FP32_TFLOPS_NOMINAL, "nominal fp32 FFMA (152 SMs x 128 lanes x 2 x 2.07 GHz)"
    t_c, t_m = fl / (pk * 1e12), by / (peaks["hbm_gbs"] * 1e9)
    return fl, by, max(t_c, t_m), ("hbm" if t_m >= t_c else ("tensor" if w.dtype == "bf16" else "alu")), pk, src


def time_steps(gdn, w, d, ws, run, steps, stream, flush, scrub, prof_every):
    """Device seconds of `steps` back-to-back steps (CUDA events on the
    launching stream), with the library's per-launch event pairs on every
    prof_every-th step. Inputs that fit in L2 get a write of twice the L2
    size before every step, outside that step's own events."""
    import torch
    prof = lambda i: gdn.profile_enable(prof_every > 0 and i % prof_every == 0)
    if not flush:
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(steps):
            prof(i)
            run(gdn, w, d, ws)
        b.record(stream)
        torch.cuda.synchronize()
        sec = a.elapsed_time(b) / 1e3
    else:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for i, (ea, eb) in enumerate(evs):
            scrub.zero_()
            ea.record(stream)
            prof(i)
            run(gdn, w, d, ws)
            eb.record(stream)
        torch.cuda.synchronize()
        sec = sum(ea.elapsed_time(eb) for ea, eb in evs) / 1e3
    gdn.profile_enable(False)
    return sec


def dominant_roofline(w, per_kernel, prof_steps, by, peaks, peak_src, workload_name, T_override):
    """The `roofline` object for the kernel with the largest device time:
    achieved = the path's algorithmic bytes per launch (inputs read once,
    outputs written once, divided over the launches of that kernel in one
    step) / its average launch time."""
    if not per_kernel:
        return None
    name, (ms_tot, n) = max(per_kernel.items(), key=lambda kv: kv[1][0])
    avg_s = ms_tot / 1e3 / n
    per_step = n / max(1, prof_steps)
    alg = by / per_step
    ach = alg / avg_s / 1e9
    return {"bound": "hbm", "kernel": name, "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": ach / peaks["hbm_gbs"],
            "traffic": measured_traffic(name, workload_name) if T_override is None else None,
            "algorithmic_bytes": alg,
            "algorithmic_bytes_basis": "path minimum per launch: inputs read once, outputs "
                                       "written once, h0 / h_final once, no intermediates",
            "launches_per_step": per_step,
            "kernel_image_bytes": kernel_bytes(w, name),
            "avg_launch_us": avg_s * 1e6, "peak_source": f"{peak_src} hbm_gbs"}


def sweep_configs(gdn, dev, stream, peaks, headline, rank, steps=10, warmup=3):
    """Every workload of the benchmark statement timed the same way as the
    headline (one entry per workload; the headline's own entry repeats its
    numbers): ms per step, tokens/s, algorithmic TFLOP/s, the path roofline
    fraction and the per-kernel times. The 256-token fp32 workload also gets
    the fraction of a CUDA-graph replay of 64 back-to-back calls."""
    import torch
    out = {}
    for name in CONFIGS:
        if name == headline["config"]["workload"]:
            out[name] = {k: headline[k] for k in ("ms_per_step", "value", "tflops")}
            out[name]["tokens_per_s"] = out[name].pop("value")
            out[name]["path_frac"] = headline["path_roofline"]["frac"]
            out[name]["kernels_us"] = {k: v["avg_us"] for k, v in headline["kernels"].items()}
            out[name]["steps"] = headline["steps"]
            continue
        w = workloads.build(name, seed=rank)
        w = resolve_segments(gdn, w, dev)
        d = device_inputs(w, dev)
        ws = workspace_for(gdn, w, dev)
        _, flush = config_of(w, name, 1)
        scrub = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if flush else None
        for _ in range(warmup):
            run_step(gdn, w, d, ws)
        torch.cuda.synchronize()
        gdn.profile_collect()
        sec = time_steps(gdn, w, d, ws, run_step, steps, stream, flush, scrub, 0)
        # per-kernel times from a second run with an event pair around every launch
        time_steps(gdn, w, d, ws, run_step, min(steps, 5), stream, flush, scrub, 1)
        per_kernel = gdn.profile_collect()
        step_s = sec / steps
        fl, by, roof_t, bound, pk, src = path_roof(w, peaks)
        e = {"ms_per_step": step_s * 1e3, "tokens_per_s": workload_tokens(w) / step_s,
             "tflops": fl / step_s / 1e12, "path_frac": roof_t / step_s, "path_roofline_us": roof_t * 1e6,
             "bound": bound, "compute_peak_tflops": pk, "compute_peak_source": src,
             "kernels_us": {k: v[0] / v[1] * 1e3 for k, v in per_kernel.items()},
             "steps": steps, "l2": "flushed before every step" if flush else "inputs larger than L2",
             "kernel_timing": "per-launch event pairs in a separate run of the same steps"}
        if w.dtype != "bf16":
            g = graph_replay(gdn, w, d, ws, 64, fl, by, {**peaks, "bf16_tflops": pk})
            e["graph_us_per_call"] = g["us_per_call"]
            e["path_frac_graph"] = roof_t / (g["us_per_call"] * 1e-6)
            e["graph_note"] = "64 back-to-back calls in one CUDA graph, warm L2"
        out[name] = e
        del d, ws, scrub
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the side-by-side timing of every benchmark workload")
    ap.add_argument("--T", type=int, default=None,
                    help="override the token count of a dense workload (smaller profiling captures)")
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd"], default="fwd",
                    help="bwd: time the gradients (gdn_chunk_bwd, forward recompute included) "
                         "of a causal workload (bf16 or fp32), or gdn_frame_bwd of a frame-causal "
                         "one, instead of the forward")
    ap.add_argument("--graph-replay", type=int, default=0,
                    help="also time N back-to-back calls captured in one CUDA graph (forward pass)")
    ap.add_argument("--fused", action="store_true",
                    help="run the bf16 scalar-gate forward as the single fused kernel "
                         "(gdn_set_fused; the split passes are the default)")
    ap.add_argument("--segment-len", type=int, default=None,
                    help="segment-parallel state passing with this many tokens per segment "
                         "(0: one pass per sequence); default: the workload's own setting")
    args = ap.parse_args()
    warmup = max(3, args.warmup)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus)))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return main_reference(args, warmup, rank, world)

    import torch
    import gated_delta_rule_18_gb300 as gdn
    from gated_delta_rule_18_gb300.build import build as build_lib
    build_lib()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    gdn.gdn_set_fused(args.fused)
    w = workloads.build(args.workload, seed=rank, T=args.T)  # each replica its own data
    if args.segment_len is not None:
        w = dataclasses.replace(w, segment_len=args.segment_len or None)
    w = resolve_segments(gdn, w, dev)
    d = device_inputs(w, dev)
    if args.pass_ == "bwd":
        if w.bidirectional and w.frame == 1:
            raise SystemExit("--pass bwd takes a causal workload (bf16 or fp32) or a frame-causal one")
        if w.dtype == "bf16":
            d["dout"] = torch.from_numpy(workloads.stored_normal(
                rank, "dout", (w.B, w.T, w.H, w.V), "bf16").bits.view(np.int16)).to(dev).view(torch.bfloat16)
        else:  # the fp32 path's backward takes an fp32 upstream gradient
            d["dout"] = torch.from_numpy(workloads.stored_normal(
                rank, "dout", (w.B, w.T, w.H, w.V), "f32").values).to(dev)
        args.no_e2e = args.no_cpu_baseline = args.no_configs = True
        if w.frame > 1:  # the frame-causal rule: prep recompute, then gdn_frame_bwd
            d["dden"] = torch.from_numpy(np.random.default_rng(rank).standard_normal(
                (w.B, w.H, w.T)).astype(np.float32)).to(dev) if w.bidirectional else None
            ws = torch.empty(gdn.gdn_frame_bwd_workspace_size(w.B, w.T, w.H, w.K, w.V, w.frame,
                                                              w.bidirectional),
                             dtype=torch.uint8, device=dev)

            def run(gdn, w, d, ws):  # the timed step of this pass
                if w.prep == "rms_relu":
                    q = gdn.gdn_prep(d["q"], mode=gdn.PREP_RMS | gdn.PREP_RELU, scale=1.0, eps=1e-5)
                    k = gdn.gdn_prep(d["k"], mode=gdn.PREP_RMS | gdn.PREP_RELU, scale=w.K ** -0.5,
                                     eps=1e-5)
                else:
                    q = gdn.gdn_prep(d["q"], mode=gdn.PREP_L2)
                    k = gdn.gdn_prep(d["k"], mode=gdn.PREP_L2)
                return gdn.gdn_frame_bwd(q, k, d["v"], d["beta"], d["g_frame"], w.frame, d["dout"],
                                         dden=d["dden"], h0=None if w.bidirectional else d["h0"],
                                         direction=2 if w.bidirectional else 0, workspace=ws)
        else:
            ws = torch.empty(gdn.gdn_bwd_workspace_size(w.B, w.T, w.H, w.K, w.V, w.n_seq,
                                                        w.cu_seqlens is not None, w.gk is not None,
                                                        fp32=w.dtype == "f32"),
                             dtype=torch.uint8, device=dev)

            def run(gdn, w, d, ws):  # the timed step of this pass
                return gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["dout"],
                                         h0=d["h0"], qk_l2norm=w.prep == "l2", workspace=ws,
                                         cu_seqlens=d.get("cu_seqlens"), gk=d.get("gk"))
    else:
        ws = workspace_for(gdn, w, dev)
        run = run_step
    stream = torch.cuda.current_stream()
    config, flush = config_of(w, args.workload, world)
    if args.fused:
        config = dict(config, path="fused single-kernel forward (opt-in)")
    scrub = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if flush else None

    sampler = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                           else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]))
    sampler.start()
    time.sleep(0.3)
    # the warm-up steps run right before the timed ones (no idle gap between)
    for _ in range(warmup):
        run(gdn, w, d, ws)
    torch.cuda.synchronize()
    gdn.profile_collect()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = gdn.launch_count()
    # the library's per-launch event pairs (the per-kernel times) are taken on
    # every PROFILE_EVERY-th timed step: an event pair waits for the kernel
    # before it to drain, which costs ~2 us per kernel boundary
    sec = time_steps(gdn, w, d, ws, run, args.steps, stream, flush, scrub, PROFILE_EVERY)
    if dist:
        dist.barrier()
    launches = gdn.launch_count() - launches0
    per_kernel = gdn.profile_collect()
    # the same step back to back right after the timed ones, until the sampled
    # window is CLOCK_SOAK_S long: the clock record covers the timed steps and
    # this run (nvidia-smi samples every 100 ms), and its step time is a
    # cross-check of the headline
    soak_steps, soak_sec, t0 = 0, 0.0, time.perf_counter()
    while time.perf_counter() - t0 < CLOCK_SOAK_S and not flush:
        n = 50
        soak_sec += time_steps(gdn, w, d, ws, run, n, stream, False, None, 0)
        soak_steps += n
    clocks = sampler.stop()
    clocks["window"] = (f"warm-up, the {args.steps} timed steps and {soak_steps} more of the same "
                        "step back to back")
    sec = max_over_ranks(sec, dist, dev)
    ms_per_step = sec / args.steps * 1e3
    tokens = workload_tokens(w)
    value = job_tokens_per_s(tokens, world, args.steps, sec)

    peaks, peak_src = load_peaks()
    step_s = sec / args.steps
    fl, by, roof_t, bound, pk, pk_src = path_roof(w, peaks)
    prof_steps = -(-args.steps // PROFILE_EVERY)

    result = {
        "metric": METRIC if args.pass_ == "fwd" else METRIC_BWD, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": config,
        "tflops": fl * world / step_s / 1e12,
        "path_roofline": {"bound": bound, "min_bytes": by, "flops": fl,
                          "roofline_ms": roof_t * 1e3, "frac": roof_t / step_s,
                          "peak_source": f"{peak_src} hbm_gbs; compute {pk_src}"},
        "roofline": dominant_roofline(w, per_kernel, prof_steps, by, peaks, peak_src,
                                      args.workload, args.T) if args.pass_ == "fwd" else None,
        "kernels_sampled": f"per-launch CUDA event pairs on every {PROFILE_EVERY}th timed step",
        "kernels": {k2: {"avg_us": v2[0] / v2[1] * 1e3, "launches": v2[1],
                         "share": v2[0] / max(1e-9, sum(x[0] for x in per_kernel.values()))}
                    for k2, v2 in per_kernel.items()},
        "gpu_launches": launches,
        "clocks": clocks,
        "impl": "ours",
    }
    if soak_steps:
        result["ms_per_step_sustained"] = soak_sec / soak_steps * 1e3
    if args.graph_replay > 0 and args.pass_ == "fwd":
        result["graph_replay"] = graph_replay(gdn, w, d, ws, args.graph_replay, fl, by, peaks)
    if not args.no_e2e:
        e2e_s, h2d, d2h = e2e_measure(gdn, w, d, ws, max(10, min(args.steps, 50)), dev)
        e2e_s = max_over_ranks(e2e_s, dist, dev)
        result["e2e"] = {"value": tokens * world / e2e_s, "unit": "tokens/s",
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                         "pipelined": "step i+1 copied in while step i computes and i-1 copies out"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tok_s, csec, cores, desc = oracle_sample(w)
        result["cpu_baseline"] = {"value": tok_s, "unit": "tokens/s", "cores": cores,
                                  "kind": "oracle", "sample": desc, "seconds": csec}
    if world == 1 and not args.no_configs and args.T is None and args.segment_len is None \
            and args.workload in CONFIGS:
        del d, ws, scrub
        torch.cuda.empty_cache()
        result["configs"] = sweep_configs(gdn, dev, stream, peaks, result, rank)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result))


def main_reference(args, warmup, rank, world):
    """The reference arm: the fp64 CPU oracle as it stands, timed on the
    host cores, each step a bounded sample of the workload (rank 0 only)."""
    if rank != 0:
        return
    w = workloads.build(args.workload, seed=0)
    for _ in range(warmup):
        oracle_sample(w)
    secs, vals = [], []
    desc, cores = "", 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        v, s, cores, desc = oracle_sample(w)
        vals.append(v)
        secs.append(s)
    wall = time.perf_counter() - t0
    value = statistics.median(vals)
    print(json.dumps({
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": warmup, "ms_per_step": wall / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(w, args.workload, world)[0],
        "impl": "reference",
        "cpu_baseline": {"kind": "oracle", "cores": cores, "sample": desc, "value": value},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


if __name__ == "__main__":
    main()
