"""gdn_chunk_fwd_noalloc: the forward for callers that cannot allocate device
memory (hosts that forbid cudaMalloc after start-up, runtimes that own all
device memory, plug-ins handed only input/output pointers). It runs the same
kernels as gdn_chunk_fwd on the library's built-in scratch buffer, so on the
same inputs it must give exactly what gdn_chunk_fwd gives with a
caller-allocated workspace, allocate nothing, and report device-side errors
through gdn_noalloc_last_device_error.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import ctypes

import numpy as np
import pytest

import workloads
from gpu_helpers import f32_dev, i32_dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    import torch
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    from gated_delta_rule_18_gb300.build import build
    build()
    import gated_delta_rule_18_gb300 as m
    return m


def _case(w):
    return dict(q=to_dev(w.q), k=to_dev(w.k), v=to_dev(w.v), beta=f32_dev(w.beta),
                g=f32_dev(w.g), gk=f32_dev(w.gk), h0=f32_dev(w.h0),
                cu_seqlens=i32_dev(w.cu_seqlens))


CASES = [
    # bf16, dense, initial and final state
    (dict(B=2, T=200, H=2, K=64, V=64, dtype="bf16", seed=21, h0_std=0.5), False),
    # bf16, variable lengths, per-key gate
    (dict(B=1, T=1 + 64 + 130, H=3, K=128, V=128, dtype="bf16", seed=22, lengths=[1, 64, 130],
          g_mu=None, gk_mu=3.0), False),
    # bf16 with the denominator column
    (dict(B=1, T=150, H=2, K=128, V=112, dtype="bf16", seed=23), True),
    # fp32, small enough for the split (chunk-parallel prep + serial) path
    (dict(B=1, T=256, H=2, K=64, V=64, dtype="f32", seed=24, h0_std=0.5), False),
    # fp32, the fused kernel
    (dict(B=20, T=130, H=2, K=64, V=64, dtype="f32", seed=25), False),
]


def _pair(gdn, w, with_den):
    """(reference via gdn_chunk_fwd, result via gdn_chunk_fwd_noalloc)."""
    import torch
    d = _case(w)
    state = w.h0 is not None or not with_den
    hf_ref = torch.empty((w.n_seq, w.H, w.K, w.V), device="cuda") if state else None
    den_ref = torch.empty((w.B, w.H, w.T), device="cuda") if with_den else None
    ref = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], g=d["g"], gk=d["gk"],
                            h0=d["h0"], cu_seqlens=d["cu_seqlens"], h_final=hf_ref, den=den_ref,
                            qk_l2norm=True)
    out = torch.full_like(ref, float("nan"))
    hf = torch.full_like(hf_ref, float("nan")) if state else None
    den = torch.full_like(den_ref, float("nan")) if with_den else None
    gdn.gdn_chunk_fwd_noalloc(d["q"], d["k"], d["v"], d["beta"], out, g=d["g"], gk=d["gk"],
                              h0=d["h0"], cu_seqlens=d["cu_seqlens"], h_final=hf, den=den,
                              qk_l2norm=True)
    torch.cuda.synchronize()
    return (ref, hf_ref, den_ref), (out, hf, den)


def test_noalloc_matches_workspace_entry_point_twice(gdn):
    """Same kernels, same inputs, another scratch address: bit-identical
    results, on two calls in a row of every case (the second call finds the
    buffer holding the first call's contents)."""
    import torch
    for spec, with_den in CASES:
        spec = dict(spec)
        B, T, H, K, V, dt = (spec.pop(x) for x in ("B", "T", "H", "K", "V", "dtype"))
        w = workloads.make(B, T, H, K, V, dt, **spec)
        for _ in range(2):
            want, got = _pair(gdn, w, with_den)
            for a, b in zip(want, got):
                if a is not None:
                    assert torch.equal(a, b), (w.name, dt, with_den)
        assert gdn.gdn_noalloc_last_device_error() == 0


def test_noalloc_allocates_nothing(gdn):
    """After a first call (which looks up the buffer's address and loads the
    kernels), a call changes neither torch's allocator counters nor the
    device's free memory."""
    import torch
    w = workloads.make(2, 300, 2, 128, 128, "bf16", seed=26, h0_std=0.5)
    d = _case(w)
    out = torch.empty((2, 300, 2, 128), dtype=torch.bfloat16, device="cuda")
    hf = torch.empty((2, 2, 128, 128), device="cuda")

    def call():
        gdn.gdn_chunk_fwd_noalloc(d["q"], d["k"], d["v"], d["beta"], out, g=d["g"], h0=d["h0"],
                                  h_final=hf, qk_l2norm=True)
    call()
    torch.cuda.synchronize()
    a0, r0 = torch.cuda.memory_allocated(), torch.cuda.memory_reserved()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == a0 and torch.cuda.memory_reserved() == r0
    assert free1 >= free0 - (1 << 20), (free0, free1)


def test_noalloc_reports_device_errors(gdn):
    """A malformed cu_seqlens (only the device sees it) is reported through
    the built-in buffer's error word; the next good call is clean."""
    import torch
    w = workloads.make(1, 100, 2, 64, 64, "bf16", seed=9, lengths=[30, 20, 50])
    d = _case(w)
    bad = i32_dev(np.array([0, 50, 30, 100], dtype=np.int32))  # not monotone
    out = torch.zeros((1, 100, 2, 64), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_chunk_fwd_noalloc(d["q"], d["k"], d["v"], d["beta"], out, g=d["g"], cu_seqlens=bad)
    L = gdn.lib()
    word = ctypes.c_int(0)
    assert L.gdn_noalloc_last_device_error(None, ctypes.byref(word)) == 9  # GDN_ERR_DEVICE
    assert word.value == 1
    assert torch.count_nonzero(out) == 0  # nothing was computed
    gdn.gdn_chunk_fwd_noalloc(d["q"], d["k"], d["v"], d["beta"], out, g=d["g"],
                              cu_seqlens=d["cu_seqlens"])
    assert gdn.gdn_noalloc_last_device_error() == 0


def test_noalloc_status_codes_match_the_workspace_entry_point(gdn):
    """Argument errors get gdn_chunk_fwd's status; a problem that passes them
    but needs more scratch than the buffer gets GDN_ERR_WORKSPACE."""
    import torch
    L = gdn.lib()
    P = ctypes.c_void_p
    x = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    f = torch.zeros(64, dtype=torch.float32, device="cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")

    def both(B, T, H, K, V, qk_dtype, v_dtype):
        qd = gdn.TensorDesc(qk_dtype, 0, T * H * K, H * K, K)
        vd = gdn.TensorDesc(v_dtype, 0, T * H * V, H * V, V)
        args = (P(x.data_ptr()), P(x.data_ptr()), qd, P(x.data_ptr()), vd, P(f.data_ptr()), None,
                P(f.data_ptr()), None, None, B, P(x.data_ptr()), vd, None, None, B, T, H, K, V, 64,
                0, 0)
        a = L.gdn_chunk_fwd(*args, P(ws.data_ptr()), ws.numel(), None)
        b = L.gdn_chunk_fwd_noalloc(*args, None)
        return a, b
    a, b = both(1, 64, 2, 64, 64, gdn.BF16, gdn.F32)  # q/k and v dtypes differ
    assert a == b == 3  # GDN_ERR_DTYPE
    a, b = both(1, 64, 2, 256, 64, gdn.BF16, gdn.BF16)  # K > 128
    assert a == b == 2  # GDN_ERR_SHAPE
    B, T, H, K, V = 1, 1 << 16, 32, 128, 128   # needs far more than the buffer
    assert gdn.gdn_workspace_size(B, T, H, K, V, B, 0, gdn.BF16, 0) > (64 << 20)
    _, b = both(B, T, H, K, V, gdn.BF16, gdn.BF16)
    assert b == 8  # GDN_ERR_WORKSPACE, nothing launched
