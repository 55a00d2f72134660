"""fp64 CPU oracle for the gated delta rule forward scan.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg may import this package; the product path (the CUDA library and
its Python binding) never does, and the two share no code.

The arithmetic lives in `gdn_oracle.c` (a plain token-by-token fp64 loop,
parallel over (sequence, head) with pthreads); this module compiles it with
gcc and marshals numpy arrays. Every function takes the STORED input values
(bf16 inputs upcast exactly) and computes in float64.

Pins that tie it to the pages and to mathematics, independently of itself,
are in tests/test_oracle_pins.py; every function here has at least one.
The gradients of the scan (`oracle.backward`) are the float64 autograd
derivative of the plain token loop, pinned to central finite differences of
the C forward above.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdn_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE fp64, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                           "-pthread", "-fno-fast-math", "-ffp-contract=off",
                           _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            lib.oracle_gdn_scan.restype = ctypes.c_int
            lib.oracle_gdn_scan.argtypes = [
                ctypes.c_int, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                P, P, P, P, P, P, P, ctypes.c_int, P, P, ctypes.c_int]
            lib.oracle_gdn_frame_scan.restype = ctypes.c_int
            lib.oracle_gdn_frame_scan.argtypes = [
                ctypes.c_int, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                P, P, P, P, P, P, ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int]
            lib.oracle_l2norm.restype = None
            lib.oracle_l2norm.argtypes = [P, ctypes.c_int64, ctypes.c_int,
                                          ctypes.c_double, P]
            lib.oracle_rmsnorm.restype = None
            lib.oracle_rmsnorm.argtypes = [P, ctypes.c_int64, ctypes.c_int,
                                           ctypes.c_double, ctypes.c_int,
                                           ctypes.c_double, P, P]
            _lib = lib
    return _lib


def _f64(x):
    return None if x is None else np.ascontiguousarray(x, dtype=np.float64)


def _ptr(x):
    return None if x is None else x.ctypes.data


def default_threads() -> int:
    return os.cpu_count() or 1


def scan(q, k, v, beta, g=None, gk=None, h0=None, cu_seqlens=None,
         reverse=False, threads=None):
    """Token-level gated delta rule.

    Dense: q, k (B, T, H, K); v (B, T, H, V); beta, g (B, T, H);
    gk (B, T, H, K); h0 (B, H, K, V) or None.
    Varlen: B == 1 and cu_seqlens (n_seq+1,) marks the sequences; h0 is then
    (n_seq, H, K, V).
    Returns (out (B, T, H, V), h_final (n_seq, H, K, V)) in float64.
    """
    q, k, v, beta, g, gk, h0 = map(_f64, (q, k, v, beta, g, gk, h0))
    B, T, H, K = q.shape
    V = v.shape[-1]
    if cu_seqlens is None:
        row0 = np.arange(B, dtype=np.int64) * T
        lens = np.full(B, T, dtype=np.int64)
    else:
        assert B == 1
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        row0 = np.ascontiguousarray(cu[:-1])
        lens = np.ascontiguousarray(cu[1:] - cu[:-1])
    n_seq = len(lens)
    out = np.zeros((B, T, H, V), dtype=np.float64)
    hf = np.zeros((n_seq, H, K, V), dtype=np.float64)
    rc = _load().oracle_gdn_scan(
        n_seq, _ptr(row0), _ptr(lens), H, K, V, _ptr(q), _ptr(k), _ptr(v),
        _ptr(g), _ptr(gk), _ptr(beta), _ptr(h0), int(bool(reverse)), _ptr(out),
        _ptr(hf), int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_gdn_scan failed with status {rc}")
    return out, hf


def frame_scan(q, k, v, beta, g_frame, frame, h0=None, reverse=False, threads=None):
    """Frame-causal rule (see `oracle_gdn_frame_scan` in gdn_oracle.c): frames
    of `frame` tokens share one pre-frame state for their predictions and
    output from the post-frame state. Dense only: q, k (B, T, H, K); v
    (B, T, H, V); beta (B, T, H); g_frame (B, T // frame, H) log decays;
    h0 (B, H, K, V) or None. Returns (out, h_final) in float64."""
    q, k, v, beta, g_frame, h0 = map(_f64, (q, k, v, beta, g_frame, h0))
    B, T, H, K = q.shape
    V = v.shape[-1]
    assert T % frame == 0 and g_frame.shape == (B, T // frame, H)
    row0 = np.arange(B, dtype=np.int64) * T
    lens = np.full(B, T, dtype=np.int64)
    out = np.zeros((B, T, H, V), dtype=np.float64)
    hf = np.zeros((B, H, K, V), dtype=np.float64)
    rc = _load().oracle_gdn_frame_scan(
        B, _ptr(row0), _ptr(lens), H, K, V, _ptr(q), _ptr(k), _ptr(v), _ptr(g_frame),
        _ptr(beta), _ptr(h0), int(frame), int(bool(reverse)), _ptr(out), _ptr(hf),
        int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_gdn_frame_scan failed with status {rc}")
    return out, hf


def frame_den(q, k, beta, g_frame, frame, reverse=False, threads=None):
    """Denominator of the frame-causal rule: the same recurrence with V = 1,
    v = 1. Returns (B, H, T) float64."""
    B, T, H, _ = np.shape(q)
    ones = np.ones((B, T, H, 1), dtype=np.float64)
    out, _ = frame_scan(q, k, ones, beta, g_frame, frame, reverse=reverse, threads=threads)
    return np.ascontiguousarray(out[..., 0].transpose(0, 2, 1))


def den(q, k, beta, g=None, gk=None, cu_seqlens=None, reverse=False,
        threads=None, z0=None, with_state=False):
    """Denominator scan: the same recurrence with V = 1 and v = 1
    (SANA `fused_gdn.py` page, `_fused_gdn_kernel` z-state). z0: the z
    state (n_seq, H, K) the scan starts from (init_state_z), or None for
    zero. Returns (B, H, T) float64, and with with_state also the final z
    state (n_seq, H, K)."""
    B, T, H, _ = np.shape(q)
    ones = np.ones((B, T, H, 1), dtype=np.float64)
    h0 = None if z0 is None else np.asarray(z0, dtype=np.float64)[..., None]
    out, zf = scan(q, k, ones, beta, g=g, gk=gk, h0=h0, cu_seqlens=cu_seqlens,
                   reverse=reverse, threads=threads)
    d = np.ascontiguousarray(out[..., 0].transpose(0, 2, 1))
    return (d, np.ascontiguousarray(zf[..., 0])) if with_state else d


def state_summary(k, v, beta, segment_len, g=None, gk=None, threads=None):
    """Affine summary of every segment of every sequence (hyper-parallel
    coverage_diff page, `kda_state_summary_forward_from_prepared` returning
    state_ext and transition): over segment s (tokens s*L .. s*L+L-1, the last
    one ragged) the causal token recurrence maps the entering state h to
    M_s h + E_s. The recurrence is linear in the state with v entering only
    additively, so E_s is the scan's final state from h = 0, and column j of
    M_s is the final state of the same scan with v = 0 from h = e_j.
    Dense only: k (B, T, H, K); v (B, T, H, V); beta, g (B, T, H); gk
    (B, T, H, K). Returns (ext (n_seg, B, H, K, V), tr (n_seg, B, H, K, K))
    in float64."""
    k, v, beta, g, gk = map(_f64, (k, v, beta, g, gk))
    B, T, H, K = k.shape
    V = v.shape[-1]
    L = int(segment_len)
    n_seg = -(-T // L)
    ext = np.zeros((n_seg, B, H, K, V))
    tr = np.zeros((n_seg, B, H, K, K))
    eye = np.ascontiguousarray(np.broadcast_to(np.eye(K), (B, H, K, K)))
    for s in range(n_seg):
        sl = slice(s * L, min((s + 1) * L, T))
        ks, vs, bs = k[:, sl], v[:, sl], beta[:, sl]
        gs = None if g is None else g[:, sl]
        gks = None if gk is None else gk[:, sl]
        _, ext[s] = scan(ks, ks, vs, bs, g=gs, gk=gks, threads=threads)
        _, tr[s] = scan(ks, ks, np.zeros(ks.shape[:3] + (K,)), bs, g=gs, gk=gks, h0=eye,
                        threads=threads)
    return ext, tr


def l2norm(x, eps=1e-6):
    """Per-row L2 normalisation over the last dim: x / sqrt(sum x^2 + eps)."""
    x = _f64(x)
    D = x.shape[-1]
    y = np.empty_like(x)
    _load().oracle_l2norm(_ptr(x), x.size // D, D, float(eps), _ptr(y))
    return y


def rmsnorm_channels(x, eps=1e-5, relu=False, scale=1.0):
    """Full-channel RMSNorm of x (B, T, H, D) over the H*D channels of each
    token, then optional ReLU, then * scale. Returns (y, inv_rms (B, T))."""
    x = _f64(x)
    B, T, H, D = x.shape
    y = np.empty_like(x)
    inv = np.empty((B, T), dtype=np.float64)
    _load().oracle_rmsnorm(_ptr(x), B * T, H * D, float(eps), int(bool(relu)),
                           float(scale), _ptr(y), _ptr(inv))
    return y, inv


def merge(num, den_, gate=None, eps=1e-6):
    """The bidirectional merge (SANA `fused_gdn.py` page, `fused_bigdn_func`
    and `_fused_bidi_merge_kernel` with its optional gate):
    out = num / (den + eps) * silu(gate), silu(x) = x / (1 + e^{-x}).
    num, gate: (B, T, H, V); den: (B, H, T). Returns float64 (B, T, H, V)."""
    num = _f64(num)
    d = np.asarray(den_, dtype=np.float64).transpose(0, 2, 1)[..., None]
    out = num / (d + eps)
    if gate is not None:
        x = _f64(gate)
        with np.errstate(over="ignore"):
            out = out * (x / (1.0 + np.exp(-x)))
    return out


def forward(w, threads=None):
    """The whole forward of a `workloads.Workload`: prep, then the causal
    scan, or (bidirectional) the causal plus the reverse scan summed, with
    the denominator. Returns a dict of float64 arrays."""
    qv, kv, vv = w.q.values, w.k.values, w.v.values
    res = {}
    if w.prep == "l2":
        qn, kn = l2norm(qv), l2norm(kv)
    elif w.prep == "rms_relu":
        qn, res["q_inv_rms"] = rmsnorm_channels(qv, 1e-5, relu=True, scale=1.0)
        kn, res["k_inv_rms"] = rmsnorm_channels(kv, 1e-5, relu=True,
                                                scale=w.K ** -0.5)
    else:
        raise ValueError(w.prep)
    if getattr(w, "frame", 1) > 1:
        # frame-causal form (bidirectional: both directions summed, with den)
        S, gf = w.frame, w.g_frame
        of, hf = frame_scan(qn, kn, vv, w.beta, gf, S, h0=w.h0, threads=threads)
        if not w.bidirectional:
            res["out"], res["h_final"] = of, hf
            return res
        orv, _ = frame_scan(qn, kn, vv, w.beta, gf, S, reverse=True, threads=threads)
        res["out"] = of + orv
        res["den"] = (frame_den(qn, kn, w.beta, gf, S, threads=threads)
                      + frame_den(qn, kn, w.beta, gf, S, reverse=True, threads=threads))
        return res
    if not w.bidirectional:
        out, hf = scan(qn, kn, vv, w.beta, g=w.g, gk=w.gk, h0=w.h0,
                       cu_seqlens=w.cu_seqlens, threads=threads)
        res["out"], res["h_final"] = out, hf
        return res
    # the backward direction takes its own gates / beta when given (the
    # chunk-causal form of the SANA `fused_gdn.py` page: decay_bwd, beta_bwd)
    gb = w.g if getattr(w, "g_bwd", None) is None else w.g_bwd
    bb = w.beta if getattr(w, "beta_bwd", None) is None else w.beta_bwd
    of, _ = scan(qn, kn, vv, w.beta, g=w.g, gk=w.gk, cu_seqlens=w.cu_seqlens,
                 threads=threads)
    orv, _ = scan(qn, kn, vv, bb, g=gb, gk=w.gk, cu_seqlens=w.cu_seqlens,
                  reverse=True, threads=threads)
    res["out"] = of + orv
    res["den"] = (den(qn, kn, w.beta, g=w.g, gk=w.gk, cu_seqlens=w.cu_seqlens,
                      threads=threads)
                  + den(qn, kn, bb, g=gb, gk=w.gk,
                        cu_seqlens=w.cu_seqlens, reverse=True, threads=threads))
    if getattr(w, "merge", False):
        gate = None if w.gate is None else w.gate.values
        res["merged"] = merge(res["out"], res["den"], gate=gate, eps=w.eps)
    return res
