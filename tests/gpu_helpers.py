"""Helpers for the GPU parity tests: move seeded workloads to the device, run
the CUDA path through the binding, compare with the fp64 oracle."""
from __future__ import annotations

import numpy as np

TOL = {"f32": 1e-4, "bf16": 2e-2}  # max|gpu - ref| / max|ref|


def torch():
    import torch as t
    return t


def dev():
    return torch().device("cuda:0")


def to_dev(st):
    """workloads.Stored -> device tensor holding the same stored values."""
    t = torch()
    if st.dtype == "bf16":
        bits = np.ascontiguousarray(st.bits)
        return t.from_numpy(bits.view(np.int16)).to(dev()).view(t.bfloat16)
    return t.from_numpy(np.ascontiguousarray(st.values)).to(dev())


def f32_dev(a):
    if a is None:
        return None
    return torch().from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev())


def i32_dev(a):
    if a is None:
        return None
    return torch().from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev())


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite GPU output"
    scale = np.abs(ref).max()
    return float(np.abs(got - ref).max() / (scale if scale > 0 else 1.0))


def run_gpu(w, with_final_state=True):
    """Run a workloads.Workload end to end on the GPU; numpy float64 results."""
    import gated_delta_rule_18_gb300 as gdn
    t = torch()
    if w.qkv is not None:
        qkv = to_dev(w.qkv)
        q, k, v = qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2]
    else:
        q, k, v = to_dev(w.q), to_dev(w.k), to_dev(w.v)
    bw = {}
    if w.g_bwd is not None:
        bw["g"] = f32_dev(w.g_bwd)
    if w.beta_bwd is not None:
        bw["beta"] = f32_dev(w.beta_bwd)
    extra = {}
    if w.frame > 1:
        extra = dict(frame=w.frame, g_frame=f32_dev(w.g_frame))
    elif w.bidirectional and (bw or w.merge):
        extra = dict(backward=bw or None, merge=w.merge, eps=w.eps,
                     gate=None if w.gate is None else to_dev(w.gate))
    if w.segment_len is not None:
        extra["segment_len"] = w.segment_len
    res = gdn.gdn_forward(q, k, v, f32_dev(w.beta), g=f32_dev(w.g), gk=f32_dev(w.gk),
                          h0=f32_dev(w.h0), cu_seqlens=i32_dev(w.cu_seqlens), prep=w.prep,
                          bidirectional=w.bidirectional,
                          with_final_state=with_final_state and not w.bidirectional, **extra)
    t.cuda.synchronize()
    return {k2: v2.double().cpu().numpy() for k2, v2 in res.items()}
