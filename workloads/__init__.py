"""Seeded synthetic inputs for the gated delta rule forward scan.

This module is shared by the tests, the benchmark and the smoke check. It
draws random numbers and encodes them into storage types; it holds none of
the scan's arithmetic (no normalisation, no recurrence, no gating maths), so
that the fp64 oracle and the CUDA path both consume identical stored values
without sharing any computation.

Recipe (every workload, seed 0 unless stated):
  * q, k, v ~ N(0, 1), drawn in float32 and rounded to the storage dtype
    (bf16 by round-to-nearest-even, or kept in fp32).
  * beta = sigmoid(N(0, 1)) per (token, head), stored fp32.
  * g = log(sigmoid(N(mu, 1))) per (token, head), stored fp32 (mu = 3, or 4
    for the video workload); for the per-key workload gk has the same law per
    (token, head, key channel) with mu = 4.
  * varlen lengths: integers uniform on [128, 8192] inclusive; initial states
    h0 ~ N(0, 0.02^2) per sequence.
Each tensor gets its own generator seeded by (seed, tensor id, block index)
so that tensors are independent of one another and of the thread count used
to fill them; numpy's PCG64 is platform independent, so the Arm GPU host and
the x86 build host draw identical values.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os

import numpy as np

BLOCK = 1 << 22  # elements per independently seeded block

_TENSOR_IDS = {"q": 1, "k": 2, "v": 3, "beta": 4, "g": 5, "gk": 6, "h0": 7,
               "lens": 8, "qkv": 9, "gate": 10, "g_frame": 11, "dout": 12}


def _normal_fill(seed: int, name: str, n: int, mu: float, sigma: float,
                 out: np.ndarray, encode) -> np.ndarray:
    """Fill `out` (length n) with encode(N(mu, sigma^2) float32 draws), block
    by block; each block has its own generator seeded (seed, tensor, block)."""
    tid = _TENSOR_IDS[name]
    nblk = (n + BLOCK - 1) // BLOCK

    def fill(b: int) -> None:
        lo, hi = b * BLOCK, min(n, (b + 1) * BLOCK)
        rng = np.random.default_rng([seed, tid, b])
        x = rng.standard_normal(hi - lo, dtype=np.float32)
        if sigma != 1.0:
            x *= np.float32(sigma)
        if mu != 0.0:
            x += np.float32(mu)
        out[lo:hi] = encode(x)

    if nblk <= 1:
        for b in range(nblk):
            fill(b)
    else:
        workers = min(nblk, os.cpu_count() or 1, 16)
        with _cf.ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, range(nblk)))
    return out


def _normal_f32(seed: int, name: str, n: int, mu: float = 0.0,
                sigma: float = 1.0) -> np.ndarray:
    """n draws of N(mu, sigma^2) as float32."""
    return _normal_fill(seed, name, n, mu, sigma, np.empty(n, dtype=np.float32),
                        lambda x: x)


def bf16_round_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even.

    Inputs here are finite; NaN handling is not needed."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits).astype(np.uint32) << np.uint32(16)).view(np.float32)


class Stored:
    """A tensor as stored: fp32 data, or bf16 bit patterns (uint16).

    `values` is the exact float32 view of what is stored (computed on demand
    for bf16, so huge tensors can be sliced before upcasting)."""

    def __init__(self, dtype: str, data: np.ndarray):
        assert dtype in ("f32", "bf16")
        self.dtype = dtype
        self._data = data

    @property
    def bits(self) -> np.ndarray:
        assert self.dtype == "bf16"
        return self._data

    @property
    def values(self) -> np.ndarray:
        if self.dtype == "bf16":
            return bf16_bits_to_f32(self._data)
        return self._data

    @property
    def shape(self):
        return self._data.shape

    def take(self, index) -> "Stored":
        """The stored tensor restricted by a numpy index (no upcast)."""
        return Stored(self.dtype, np.ascontiguousarray(self._data[index]))


def stored_normal(seed: int, name: str, shape, dtype: str, mu=0.0,
                  sigma=1.0) -> Stored:
    n = int(np.prod(shape))
    if dtype == "bf16":
        out = _normal_fill(seed, name, n, mu, sigma, np.empty(n, dtype=np.uint16),
                           bf16_round_bits)
        return Stored("bf16", out.reshape(shape))
    if dtype == "f32":
        return Stored("f32", _normal_f32(seed, name, n, mu, sigma).reshape(shape))
    raise ValueError(dtype)


def _sigmoid(x: np.ndarray) -> np.ndarray:
    xd = x.astype(np.float64)
    return (1.0 / (1.0 + np.exp(-xd))).astype(np.float32)


def _log_sigmoid(x: np.ndarray) -> np.ndarray:
    xd = x.astype(np.float64)
    with np.errstate(over="ignore"):
        y = np.where(xd > 0, -np.log1p(np.exp(-xd)), xd - np.log1p(np.exp(xd)))
    return y.astype(np.float32)


def sigmoid_normal(seed: int, name: str, shape, mu: float) -> np.ndarray:
    """sigmoid(N(mu,1)) as float32 (computed in float64 then rounded)."""
    n = int(np.prod(shape))
    return _normal_fill(seed, name, n, mu, 1.0, np.empty(n, dtype=np.float32),
                        _sigmoid).reshape(shape)


def log_sigmoid_normal(seed: int, name: str, shape, mu: float) -> np.ndarray:
    """log(sigmoid(N(mu,1))) = -log1p(exp(-x)) as float32."""
    n = int(np.prod(shape))
    return _normal_fill(seed, name, n, mu, 1.0, np.empty(n, dtype=np.float32),
                        _log_sigmoid).reshape(shape)


@dataclasses.dataclass
class Workload:
    """One forward problem. Layouts (row-major):
    q, k: (B, T, H, K) raw (un-normalised) values; v: (B, T, H, V);
    beta, g: (B, T, H); gk: (B, T, H, K); h0: (n_seq, H, K, V);
    cu_seqlens: (n_seq + 1,) int32 when varlen (then B == 1).
    For the video workload `qkv` (B, T, 3, H, D) holds q, k, v interleaved and
    q, k, v are views into it."""
    name: str
    B: int
    T: int
    H: int
    K: int
    V: int
    dtype: str
    q: Stored
    k: Stored
    v: Stored
    beta: np.ndarray
    g: np.ndarray | None = None
    gk: np.ndarray | None = None
    h0: np.ndarray | None = None
    cu_seqlens: np.ndarray | None = None
    qkv: Stored | None = None
    prep: str = "l2"          # "l2" | "rms_relu"
    bidirectional: bool = False
    chunk: int = 64
    # chunk-causal bidirectional form: gates / beta of the backward direction
    # (None: the forward ones), and the merge out = num / (den + eps) *
    # silu(gate) with `gate` (B, T, H, V)
    g_bwd: np.ndarray | None = None
    beta_bwd: np.ndarray | None = None
    merge: bool = False
    gate: Stored | None = None
    eps: float = 1e-6
    # frame-causal form: `frame` tokens per frame share the pre-frame state;
    # one log-decay per frame, g_frame (B, T // frame, H) (then g is None)
    frame: int = 1
    g_frame: np.ndarray | None = None
    # how the GPU path walks each sequence (same result): segment-parallel
    # state passing with segments of this many tokens, "auto" to let the
    # library pick for the device, or None for one pass per sequence
    segment_len: int | str | None = None

    @property
    def n_seq(self) -> int:
        return self.B if self.cu_seqlens is None else len(self.cu_seqlens) - 1

    @property
    def tokens(self) -> int:
        return self.B * self.T


def _vary_lengths(seed: int, n_seq: int, lo: int, hi: int) -> np.ndarray:
    rng = np.random.default_rng([seed, _TENSOR_IDS["lens"], 0])
    return rng.integers(lo, hi + 1, size=n_seq)


def make(B: int, T: int, H: int, K: int, V: int, dtype: str = "bf16", *,
         seed: int = 0, g_mu: float | None = 3.0, gk_mu: float | None = None,
         h0_std: float | None = None, lengths=None, name: str = "custom",
         chunk: int = 64, segment_len: int | str | None = None) -> Workload:
    """A causal workload with q, k, v ~ N(0,1), beta = sigmoid(N(0,1)) and a
    scalar gate (g_mu) or a per-key gate (gk_mu). `lengths` (list of ints)
    makes it varlen: B must be 1 and T == sum(lengths)."""
    cu = None
    n_seq = B
    if lengths is not None:
        lengths = [int(x) for x in lengths]
        assert B == 1 and T == sum(lengths)
        cu = np.zeros(len(lengths) + 1, dtype=np.int32)
        cu[1:] = np.cumsum(lengths)
        n_seq = len(lengths)
    q = stored_normal(seed, "q", (B, T, H, K), dtype)
    k = stored_normal(seed, "k", (B, T, H, K), dtype)
    v = stored_normal(seed, "v", (B, T, H, V), dtype)
    beta = sigmoid_normal(seed, "beta", (B, T, H), 0.0)
    g = log_sigmoid_normal(seed, "g", (B, T, H), g_mu) if g_mu is not None else None
    gk = log_sigmoid_normal(seed, "gk", (B, T, H, K), gk_mu) if gk_mu is not None else None
    h0 = None
    if h0_std is not None:
        h0 = _normal_f32(seed, "h0", n_seq * H * K * V, 0.0, h0_std).reshape(n_seq, H, K, V)
    return Workload(name, B, T, H, K, V, dtype, q, k, v, beta, g, gk, h0, cu,
                    chunk=chunk, segment_len=segment_len)


def make_video(B: int, N: int, H: int, D: int, *, seed: int = 0,
               g_mu: float = 4.0, name: str = "video", reset_every: int | None = None,
               merge: bool = False, frame: int = 1) -> Workload:
    """Interleaved qkv (B, N, 3, H, D) ~ N(0,1) bf16, bidirectional, with the
    full-channel RMSNorm + ReLU + k-scale prep.

    reset_every = R makes it chunk-causal: the backward direction's log-gate
    is -inf and its beta 0 at tokens R, 2R, ..., so that a token's backward
    state holds only the later tokens of its own R-token chunk. merge adds
    out = num / (den + eps) * silu(gate), gate (B, N, H, D) ~ N(0,1) bf16.
    frame = S > 1 makes it frame-causal: frames of S tokens, one log-decay per
    frame and head, log sigmoid(N(g_mu, 1)) (B, N // S, H)."""
    qkv = stored_normal(seed, "qkv", (B, N, 3, H, D), "bf16")
    beta = sigmoid_normal(seed, "beta", (B, N, H), 0.0)
    g = log_sigmoid_normal(seed, "g", (B, N, H), g_mu)
    g_bwd = beta_bwd = None
    if reset_every:
        g_bwd, beta_bwd = g.copy(), beta.copy()
        g_bwd[:, reset_every::reset_every, :] = -np.inf
        beta_bwd[:, reset_every::reset_every, :] = 0.0
    gate = stored_normal(seed, "gate", (B, N, H, D), "bf16") if merge else None
    g_frame = None
    if frame > 1:
        assert N % frame == 0
        g, g_frame = None, log_sigmoid_normal(seed, "g_frame", (B, N // frame, H), g_mu)

    def part(i):
        return qkv.take((slice(None), slice(None), i))
    return Workload(name, B, N, H, D, D, "bf16", part(0), part(1), part(2),
                    beta, g, qkv=qkv, prep="rms_relu", bidirectional=True,
                    g_bwd=g_bwd, beta_bwd=beta_bwd, merge=merge, gate=gate,
                    frame=frame, g_frame=g_frame)


# The five workloads, named by what they are.
WORKLOADS = {
    "causal_f32_b1h2t256d64": dict(kind="dense", B=1, T=256, H=2, K=64, V=64,
                                   dtype="f32", g_mu=3.0),
    # 64 independent problems of the 256-token fp32 shape in one launch
    "causal_f32_b64h2t256d64": dict(kind="dense", B=64, T=256, H=2, K=64, V=64,
                                    dtype="f32", g_mu=3.0),
    "causal_bf16_b4h16t4096d128": dict(kind="dense", B=4, T=4096, H=16, K=128,
                                       V=128, dtype="bf16", g_mu=3.0),
    "bidir_video_b2h16n8192d112": dict(kind="video", B=2, N=8192, H=16, D=112),
    "chunkcausal_merge_video_b2h16n8192d112": dict(kind="video", B=2, N=8192, H=16,
                                                   D=112, reset_every=1024, merge=True),
    "frame_video_b2h16f8s1024d112": dict(kind="video", B=2, N=8192, H=16, D=112,
                                         frame=1024),
    "varlen_bf16_64seq_h32d128": dict(kind="varlen", n_seq=64, lo=128, hi=8192,
                                      H=32, K=128, V=128, h0_std=0.02),
    "gk_bf16_b1h32t65536k128v256": dict(kind="dense", B=1, T=65536, H=32,
                                        K=128, V=256, dtype="bf16", g_mu=None,
                                        gk_mu=4.0),
    # one long sequence of few heads, carried in from a prefix (h0) and out
    # (h_final): segment-parallel state passing
    "seg_long_bf16_b1h4t65536d128": dict(kind="dense", B=1, T=65536, H=4, K=128,
                                         V=128, dtype="bf16", g_mu=3.0, h0_std=0.02,
                                         segment_len="auto"),
}


def varlen_lengths(seed: int = 0, n_seq: int = 64, lo: int = 128,
                   hi: int = 8192) -> list[int]:
    return [int(x) for x in _vary_lengths(seed, n_seq, lo, hi)]


def build(name: str, seed: int = 0, T: int | None = None) -> Workload:
    """The named workload; `T` overrides the token count of the dense and
    video workloads (same recipe, fewer tokens)."""
    spec = dict(WORKLOADS[name])
    kind = spec.pop("kind")
    if T is not None:
        if kind == "dense":
            spec["T"] = T
        elif kind == "video":
            spec["N"] = T
        else:
            raise ValueError("T override applies to dense and video workloads")
    if kind == "dense":
        return make(spec["B"], spec["T"], spec["H"], spec["K"], spec["V"],
                    spec["dtype"], seed=seed, g_mu=spec.get("g_mu"),
                    gk_mu=spec.get("gk_mu"), h0_std=spec.get("h0_std"), name=name,
                    segment_len=spec.get("segment_len"))
    if kind == "video":
        return make_video(spec["B"], spec["N"], spec["H"], spec["D"], seed=seed,
                          name=name, reset_every=spec.get("reset_every"),
                          merge=spec.get("merge", False), frame=spec.get("frame", 1))
    if kind == "varlen":
        lens = varlen_lengths(seed, spec["n_seq"], spec["lo"], spec["hi"])
        return make(1, sum(lens), spec["H"], spec["K"], spec["V"], "bf16",
                    seed=seed, g_mu=3.0, h0_std=spec["h0_std"], lengths=lens,
                    name=name)
    raise ValueError(kind)
