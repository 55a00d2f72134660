"""gdn_chunk_fwd_noalloc: the forward for callers that cannot allocate device
memory (hosts that forbid cudaMalloc after start-up, runtimes that own all
device memory, plug-ins handed only input/output pointers). It runs on the
library's built-in scratch buffer and must give what gdn_chunk_fwd gives with
a caller-allocated workspace.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import ctypes

import numpy as np
import pytest

import workloads
from gpu_helpers import TOL, f32_dev, i32_dev, rel_err, to_dev

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
    d = dict(q=to_dev(w.q), k=to_dev(w.k), v=to_dev(w.v), beta=f32_dev(w.beta),
             g=f32_dev(w.g), gk=f32_dev(w.gk), h0=f32_dev(w.h0),
             cu_seqlens=i32_dev(w.cu_seqlens))
    return d


def test_noalloc_matches_workspace_entry_point_twice(gdn):
    import torch
    cases = [
        workloads.make(2, 200, 2, 64, 64, "bf16", seed=21, h0_std=0.5),
        workloads.make(1, 1 + 64 + 130, 3, 128, 128, "bf16", seed=22, lengths=[1, 64, 130],
                       g_mu=None, gk_mu=3.0),
    ]
    for w in cases:  # two calls in a row, different shapes and contents
        d = _case(w)
        n_seq = w.n_seq
        hf_ref = torch.empty((n_seq, w.H, w.K, w.V), device="cuda")
        ref = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], g=d["g"], gk=d["gk"],
                                h0=d["h0"], cu_seqlens=d["cu_seqlens"], h_final=hf_ref,
                                qk_l2norm=True)
        out = torch.full_like(ref, float("nan"))
        hf = torch.full_like(hf_ref, float("nan"))
        gdn.gdn_chunk_fwd_noalloc(d["q"], d["k"], d["v"], d["beta"], out, g=d["g"], gk=d["gk"],
                                  h0=d["h0"], cu_seqlens=d["cu_seqlens"], h_final=hf,
                                  qk_l2norm=True)
        torch.cuda.synchronize()
        assert rel_err(out.double().cpu().numpy(), ref.double().cpu().numpy()) <= TOL["bf16"]
        assert rel_err(hf.double().cpu().numpy(), hf_ref.double().cpu().numpy()) <= TOL["bf16"]


def test_noalloc_rejects_problems_larger_than_its_buffer(gdn):
    import torch
    L = gdn.lib()
    B, T, H, K, V = 1, 1 << 16, 32, 128, 128   # needs far more than the buffer
    assert gdn.gdn_workspace_size(B, T, H, K, V, B, 0, gdn.BF16, 0) > (64 << 20)
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    f = torch.zeros(16, dtype=torch.float32, device="cuda")
    desc = gdn.TensorDesc(gdn.BF16, 0, T * H * K, H * K, K)
    P = ctypes.c_void_p
    st = L.gdn_chunk_fwd_noalloc(P(x.data_ptr()), P(x.data_ptr()), desc, P(x.data_ptr()), desc,
                                 P(f.data_ptr()), None, P(f.data_ptr()), None, None, B,
                                 P(x.data_ptr()), desc, None, None, B, T, H, K, V, 64, 0, 0,
                                 None)
    assert st == 8  # GDN_ERR_WORKSPACE, nothing launched
