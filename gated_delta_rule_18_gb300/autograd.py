"""torch.autograd functions over the library's forward and backward calls.

Each function's forward runs the CUDA forward through the C ABI; its
backward runs the matching gradient kernels (gdn_chunk_bwd, gdn_frame_bwd,
gdn_merge_bwd, gdn_prep_bwd).
Nothing here computes on its own: the wrappers marshal tensors and sum the
two directions' gradients.

The gradient kernels take the upstream gradient of the output in the
inputs' precision: for bf16 inputs an fp32 upstream gradient is rounded to
bf16 first; fp32 inputs (the fp32 path) keep it in fp32.
"""
from __future__ import annotations

import torch

from . import (PREP_RELU, PREP_RMS, gdn_chunk_bwd, gdn_chunk_fwd, gdn_chunk_fwd_bidir, gdn_frame_bwd,
               gdn_frame_fwd, gdn_merge, gdn_merge_bwd, gdn_prep, gdn_prep_bwd)


def _bf16(t):
    return None if t is None else t.to(torch.bfloat16).contiguous()


class _ChunkGDR(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, beta, g, gk, h0, cu_seqlens, reverse, qk_l2norm, final_state):
        n_seq = q.shape[0] if cu_seqlens is None else cu_seqlens.numel() - 1
        H, K, V = q.shape[2], q.shape[3], v.shape[3]
        hf = (torch.empty((n_seq, H, K, V), dtype=torch.float32, device=q.device)
              if final_state else None)
        o = gdn_chunk_fwd(q, k, v, beta, g=g, gk=gk, h0=h0, cu_seqlens=cu_seqlens, h_final=hf,
                          reverse=reverse, qk_l2norm=qk_l2norm)
        ctx.save_for_backward(q, k, v, beta, g, gk, h0, cu_seqlens)
        ctx.reverse, ctx.qk_l2norm = reverse, qk_l2norm
        return o, hf

    @staticmethod
    def backward(ctx, do, dhf):
        q, k, v, beta, g, gk, h0, cu_seqlens = ctx.saved_tensors
        want_h0 = h0 is not None and ctx.needs_input_grad[6]
        do = do.float().contiguous() if q.dtype == torch.float32 else _bf16(do)
        res = gdn_chunk_bwd(q, k, v, beta, g, do, h0=h0,
                            dh_final=None if dhf is None else dhf.float().contiguous(),
                            reverse=ctx.reverse, qk_l2norm=ctx.qk_l2norm, with_dh0=want_h0,
                            gk=gk, cu_seqlens=cu_seqlens)
        dg = res["dg"]
        return (res["dq"].to(q.dtype), res["dk"].to(k.dtype), res["dv"].to(v.dtype), res["dbeta"],
                None if gk is not None else dg, dg if gk is not None else None, res.get("dh0"),
                None, None, None, None)


def chunk_gated_delta_rule(q, k, v, beta, g=None, gk=None, initial_state=None,
                           output_final_state=False, cu_seqlens=None, reverse=False,
                           use_qk_l2norm=True):
    """One direction of the chunked gated delta rule, differentiable in q, k,
    v, beta, g (or the per-key gk) and initial_state. Shapes and meanings as
    gdn_chunk_fwd: q, k (B, T, H, K), v (B, T, H, V) bf16 (or all fp32: the
    fp32 path and its backward); beta, g (B, T, H)
    fp32; gk (B, T, H, K) fp32; initial_state (n_seq, H, K, V) fp32;
    cu_seqlens int32 (n_seq + 1) with B == 1. use_qk_l2norm normalises q and
    k per (token, head) inside the kernels. Returns (o, final_state or None)."""
    return _ChunkGDR.apply(q, k, v, beta, g, gk, initial_state, cu_seqlens, bool(reverse),
                           bool(use_qk_l2norm), bool(output_final_state))


class _BidirMerge(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, beta, g, gk, g_bwd, beta_bwd, gate, cu_seqlens, eps, qk_l2norm):
        B, T, H = q.shape[0], q.shape[1], q.shape[2]
        den = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
        num = gdn_chunk_fwd_bidir(q, k, v, beta, g=g, gk=gk, g_bwd=g_bwd, beta_bwd=beta_bwd,
                                  cu_seqlens=cu_seqlens, den=den, qk_l2norm=qk_l2norm)
        out = gdn_merge(num, den, gate=gate, eps=eps)
        ctx.save_for_backward(q, k, v, beta, g, gk, g_bwd, beta_bwd, gate, cu_seqlens, num, den)
        ctx.eps, ctx.qk_l2norm = eps, qk_l2norm
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, beta, g, gk, g_bwd, beta_bwd, gate, cu_seqlens, num, den = ctx.saved_tensors
        m = gdn_merge_bwd(num, den, dout.float().contiguous(), gate=gate, eps=ctx.eps)
        dnum, dden = _bf16(m["dnum"]), m["dden"]
        fwd = gdn_chunk_bwd(q, k, v, beta, g, dnum, qk_l2norm=ctx.qk_l2norm, with_dh0=False,
                            cu_seqlens=cu_seqlens, dden=dden, gk=gk)
        rev = gdn_chunk_bwd(q, k, v, beta if beta_bwd is None else beta_bwd,
                            g if g_bwd is None else g_bwd, dnum, reverse=True,
                            qk_l2norm=ctx.qk_l2norm, with_dh0=False, cu_seqlens=cu_seqlens,
                            dden=dden, gk=gk)
        dq = (fwd["dq"] + rev["dq"]).to(q.dtype)
        dk = (fwd["dk"] + rev["dk"]).to(k.dtype)
        dv = (fwd["dv"] + rev["dv"]).to(v.dtype)
        dbeta = fwd["dbeta"] if beta_bwd is not None else fwd["dbeta"] + rev["dbeta"]
        dbeta_bwd = rev["dbeta"] if beta_bwd is not None else None
        dg = fwd["dg"] if g_bwd is not None else fwd["dg"] + rev["dg"]
        dg_bwd = rev["dg"] if g_bwd is not None else None
        dgate = m.get("dgate")
        return (dq, dk, dv, dbeta, None if gk is not None else dg, dg if gk is not None else None,
                dg_bwd, dbeta_bwd, None if dgate is None else dgate.to(gate.dtype), None, None, None)


def bidirectional_gated_delta_rule(q, k, v, beta, g=None, g_bwd=None, beta_bwd=None, gate=None,
                                   cu_seqlens=None, eps=1e-6, use_qk_l2norm=True, gk=None):
    """The bidirectional form with its denominator and merge (SANA
    `fused_gdn.py` page, `fused_bigdn_func`): out = (num_fwd + num_bwd) /
    (den_fwd + den_bwd + eps) * silu(gate), differentiable in q, k, v, beta,
    g (or the per-key gk), g_bwd, beta_bwd and gate. g_bwd / beta_bwd: the
    reverse direction's own log gates / betas (the chunk-causal form; g_bwd
    with a scalar gate only), or None for g / beta."""
    return _BidirMerge.apply(q, k, v, beta, g, gk, g_bwd, beta_bwd, gate, cu_seqlens, float(eps),
                             bool(use_qk_l2norm))


class _FrameVideo(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, beta, g_frame, gate, frame, eps, prep_eps):
        K = q.shape[3]
        B, T, H = q.shape[0], q.shape[1], q.shape[2]
        mode = PREP_RMS | PREP_RELU
        qn = gdn_prep(q, mode=mode, scale=1.0, eps=prep_eps)
        kn = gdn_prep(k, mode=mode, scale=K ** -0.5, eps=prep_eps)
        den = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
        num = gdn_frame_fwd(qn, kn, v, beta, g_frame, frame, den=den, direction=2)
        out = gdn_merge(num, den, gate=gate, eps=eps)
        ctx.save_for_backward(q, k, qn, kn, v, beta, g_frame, gate, num, den)
        ctx.frame, ctx.eps, ctx.prep_eps = frame, eps, prep_eps
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, qn, kn, v, beta, g_frame, gate, num, den = ctx.saved_tensors
        K = q.shape[3]
        m = gdn_merge_bwd(num, den, dout.float().contiguous(), gate=gate, eps=ctx.eps)
        r = gdn_frame_bwd(qn, kn, v, beta, g_frame, ctx.frame, _bf16(m["dnum"]), dden=m["dden"],
                          direction=2)
        mode = PREP_RMS | PREP_RELU
        dq = gdn_prep_bwd(q, r["dq"], mode=mode, scale=1.0, eps=ctx.prep_eps)
        dk = gdn_prep_bwd(k, r["dk"], mode=mode, scale=K ** -0.5, eps=ctx.prep_eps)
        dgate = m.get("dgate")
        return (dq.to(q.dtype), dk.to(k.dtype), r["dv"].to(v.dtype), r["dbeta"], r["dg_frame"],
                None if dgate is None else dgate.to(gate.dtype), None, None, None)


def frame_video_gated_delta_rule(q, k, v, beta, g_frame, frame, gate=None, eps=1e-6, prep_eps=1e-5):
    """The video form of the SANA pages, differentiable end to end: q and k
    through the full-channel RMSNorm and ReLU (k scaled by K^-1/2), the
    frame-causal rule in both directions with its denominator (frames of
    `frame` tokens, one log decay per frame and head, g_frame (B, T / frame,
    H)), and the merge num / (den + eps) * silu(gate). q, k, v (B, T, H, D)
    bf16 (views of an interleaved qkv tensor work); beta (B, T, H) fp32."""
    return _FrameVideo.apply(q, k, v, beta, g_frame, gate, int(frame), float(eps), float(prep_eps))
