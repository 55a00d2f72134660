"""fp64 CPU oracle for the gradients of the gated delta rule scan.

TEST INFRASTRUCTURE ONLY, like the rest of `oracle/`: the tests, the smoke
check and the benchmark's CPU leg may use it; the product path never does.

The loss is L = sum(do * o) + sum(dh_final * h_final) for the token-level
recurrence (SANA `fused_gdn.py` page, `_fused_gdn_kernel`: per token, decay,
predict, correct, write; the output reads the state after the token's own
write), with optional per-(token, head) L2 normalisation of q and k (eps
1e-6) in front. The gradients are the reverse-mode derivative of that plain
token loop, taken by PyTorch autograd in float64 on the CPU: the loop below
is the definition, written out step by step, and autograd differentiates it
exactly (no chunking, no reassociation). The pages' own backward (SANA
`fused_cam_gdn.py` page, `_cam_scan_bwd_kernel`) walks the same recurrence in
reverse time with the per-step rules ds_post += q do^T, ddelta = ds_post^T k,
dv = beta ddelta, ds_pre = ds_post - k (beta ddelta)^T, ds <- e^{g} ds_pre;
autograd applies the same chain rule.

Pins (tests/test_oracle_pins.py): central finite differences of the C
oracle's forward, an independent implementation, on every input, and the
closed form of the beta = 0 case.
"""
from __future__ import annotations

import numpy as np


def _torch():
    import torch
    return torch


def _t(x):
    torch = _torch()
    return None if x is None else torch.tensor(np.asarray(x, dtype=np.float64), requires_grad=True)


def _l2(x, eps):
    return x / (x * x).sum(-1, keepdim=True).add(eps).sqrt()


def scan_torch(q, k, v, beta, g, h0=None, reverse=False, l2norm=False, eps=1e-6, gk=None):
    """The token recurrence on torch float64 tensors (differentiable).
    q, k (B, T, H, K); v (B, T, H, V); beta, g (B, T, H) or, per key, gk
    (B, T, H, K) with g None (the coverage_diff page's USE_GK: the decay
    scales the state's key rows); h0 (B, H, K, V).
    Returns (o (B, T, H, V), h_final (B, H, K, V)); reverse: the
    flip-and-shift scan (position p reads tokens p+1 .. T-1, R_{T-1} = 0)."""
    torch = _torch()
    if l2norm:
        q, k = _l2(q, eps), _l2(k, eps)
    B, T, H, K = q.shape
    V = v.shape[-1]
    S = torch.zeros(B, H, K, V, dtype=torch.float64) if h0 is None else h0
    outs = [None] * T

    def write(S, t):
        if gk is not None:
            S = torch.exp(gk[:, t])[:, :, :, None] * S                     # per-key decay
        else:
            S = torch.exp(g[:, t])[:, :, None, None] * S                   # decay
        pred = torch.einsum("bhkv,bhk->bhv", S, k[:, t])                   # S^T k
        d = beta[:, t][:, :, None] * (v[:, t] - pred)                      # correct
        return S + k[:, t][:, :, :, None] * d[:, :, None, :]               # write

    if T == 0:
        return torch.zeros(B, 0, H, V, dtype=torch.float64), S
    if not reverse:
        for t in range(T):
            S = write(S, t)
            outs[t] = torch.einsum("bhkv,bhk->bhv", S, q[:, t])
    else:
        for p in range(T - 1, -1, -1):
            outs[p] = torch.einsum("bhkv,bhk->bhv", S, q[:, p])
            S = write(S, p)
    return torch.stack(outs, dim=1), S


def scan_grad(q, k, v, beta, g, do, h0=None, dh_final=None, reverse=False, l2norm=False,
              eps=1e-6, cu_seqlens=None, gk=None):
    """Gradients of L = sum(do * o) + sum(dh_final * h_final) with respect to
    q, k, v, beta, g and h0 (raw q, k when l2norm). Returns a dict of float64
    numpy arrays: dq, dk, dv, dbeta, dg, dh0 (dh0 also when h0 is None: the
    gradient at a zero initial state), and the forward o, h_final. With a
    per-key gate gk (g None), dg is dL/dgk (B, T, H, K).
    cu_seqlens (B == 1): packed sequences, each its own recurrence from
    h0[s]; h0, dh_final and dh0 are then (n_seq, H, K, V)."""
    torch = _torch()
    B, T, H, K = np.shape(q)
    V = np.shape(v)[-1]
    if cu_seqlens is None:
        spans = [(b, 0, T) for b in range(B)]
    else:
        assert B == 1
        cu = [int(x) for x in cu_seqlens]
        spans = [(0, cu[s], cu[s + 1]) for s in range(len(cu) - 1)]
    n = len(spans)
    tq, tk, tv, tb, tg = map(_t, (q, k, v, beta, g if gk is None else gk))
    th0 = _t(np.zeros((n, H, K, V)) if h0 is None else h0)
    outs, finals = [], []
    for s, (b, a, e) in enumerate(spans):
        sl = (slice(b, b + 1), slice(a, e))
        gs = tg[sl]
        o_s, hf_s = scan_torch(tq[sl], tk[sl], tv[sl], tb[sl], None if gk is not None else gs,
                               th0[s:s + 1], reverse=reverse, l2norm=l2norm, eps=eps,
                               gk=gs if gk is not None else None)
        outs.append(o_s)
        finals.append(hf_s)
    o = torch.cat(outs, dim=1) if cu_seqlens is not None else torch.cat(outs, dim=0)
    hf = torch.cat(finals, dim=0)
    loss = (o * torch.tensor(np.asarray(do, dtype=np.float64))).sum()
    if dh_final is not None:
        loss = loss + (hf * torch.tensor(np.asarray(dh_final, dtype=np.float64))).sum()
    grads = torch.autograd.grad(loss, (tq, tk, tv, tb, tg, th0), allow_unused=True)
    names = ("dq", "dk", "dv", "dbeta", "dg", "dh0")
    shapes = (tq.shape, tk.shape, tv.shape, tb.shape, tg.shape, th0.shape)
    res = {n_: (np.zeros(s_) if gr is None else gr.detach().numpy())
           for n_, gr, s_ in zip(names, grads, shapes)}
    res["o"], res["h_final"] = o.detach().numpy(), hf.detach().numpy()
    return res


def frame_scan_torch(q, k, v, beta, g_frame, frame, h0=None, reverse=False):
    """The frame-causal rule on torch float64 tensors (differentiable), as
    the C oracle's frame scan: per frame f of `frame` tokens, S_pre =
    e^{g_f} S, then S = S_pre + sum_t beta_t k_t (v_t - S_pre^T k_t)^T, and
    every token of the frame reads the post-frame state. Reverse: frame f
    reads the state built from frames F-1 .. f+1 (each decayed by its own g
    before its write), the last frame the zero state. q, k (B, T, H, K);
    v (B, T, H, V); beta (B, T, H); g_frame (B, T // frame, H), floored at
    -30 as the forward does; h0 (B, H, K, V). Returns (o, h_final)."""
    torch = _torch()
    B, T, H, K = q.shape
    V = v.shape[-1]
    F = T // frame
    S = torch.zeros(B, H, K, V, dtype=torch.float64) if h0 is None else h0
    g = torch.clamp(g_frame, min=-30.0)

    def absorb(S, f):
        sl = slice(f * frame, (f + 1) * frame)
        Sp = torch.exp(g[:, f])[:, :, None, None] * S
        kf, vf, bf = k[:, sl], v[:, sl], beta[:, sl]                      # (B, S, H, .)
        pred = torch.einsum("bhkv,bshk->bshv", Sp, kf)
        err = bf[..., None] * (vf - pred)
        return Sp + torch.einsum("bshk,bshv->bhkv", kf, err)

    def emit(S, f):
        sl = slice(f * frame, (f + 1) * frame)
        return torch.einsum("bhkv,bshk->bshv", S, q[:, sl])

    outs = [None] * F
    for i in range(F):
        if not reverse:
            S = absorb(S, i)
            outs[i] = emit(S, i)
        else:
            if i > 0:
                S = absorb(S, F - i)
            outs[F - 1 - i] = emit(S, F - 1 - i)
    if F == 0:
        return torch.zeros(B, 0, H, V, dtype=torch.float64), S
    return torch.cat(outs, dim=1), S


def frame_grad(q, k, v, beta, g_frame, frame, do, dden=None, h0=None, dh_final=None, direction=0):
    """Gradients of L = sum(do . o) + sum(dden . den) + sum(dh_final . h_final)
    for the frame-causal rule with q, k as given (no prep): direction 0
    causal (with h0 / h_final), 1 reverse, 2 both summed (o and den are the
    sums of the two directions). den is the same rule with a ones value.
    Returns float64 numpy dq, dk, dv, dbeta, dg_frame and, for direction 0,
    dh0."""
    torch = _torch()
    B, T, H, K = np.shape(q)
    V = np.shape(v)[-1]
    tq, tk, tv, tb, tg = map(_t, (q, k, v, beta, g_frame))
    th0 = _t(np.zeros((B, H, K, V)) if h0 is None else h0)
    loss = 0.0
    for rev in ([False], [True], [False, True])[direction]:
        o, hf = frame_scan_torch(tq, tk, tv, tb, tg, frame, h0=None if rev else th0, reverse=rev)
        loss = loss + (o * torch.tensor(np.asarray(do, dtype=np.float64))).sum()
        if dden is not None:
            ones = torch.ones(B, T, H, 1, dtype=torch.float64)
            z0 = None if rev else torch.zeros(B, H, K, 1, dtype=torch.float64)
            d, _ = frame_scan_torch(tq, tk, ones, tb, tg, frame, h0=z0, reverse=rev)
            loss = loss + (d[..., 0].permute(0, 2, 1) * torch.tensor(np.asarray(dden, dtype=np.float64))).sum()
        if not rev and dh_final is not None:
            loss = loss + (hf * torch.tensor(np.asarray(dh_final, dtype=np.float64))).sum()
    grads = torch.autograd.grad(loss, (tq, tk, tv, tb, tg, th0), allow_unused=True)
    names = ("dq", "dk", "dv", "dbeta", "dg_frame", "dh0")
    shapes = (tq.shape, tk.shape, tv.shape, tb.shape, tg.shape, th0.shape)
    res = {n_: (np.zeros(s_) if gr is None else gr.detach().numpy())
           for n_, gr, s_ in zip(names, grads, shapes)}
    if direction != 0:
        res.pop("dh0")
    return res


def prep_grad(x, dy, rms=False, relu=False, scale=1.0, eps=None):
    """Gradient dL/dx of the q/k preparation y = relu?(normalised x) * scale
    for an upstream dy: rms=False normalises per (token, head) over D
    (x / sqrt(sum x^2 + eps), eps 1e-6 by default), rms=True over the H*D
    channels of a token (x / sqrt(sum x^2 / (H D) + eps), eps 1e-5; the SANA
    `fused_gdn.py` page's full-channel RMSNorm). x, dy (B, T, H, D)."""
    torch = _torch()
    tx = _t(x)
    if rms:
        B, T, H, D = tx.shape
        flat = tx.reshape(B, T, H * D)
        inv = 1.0 / torch.sqrt((flat * flat).mean(-1, keepdim=True) + (1e-5 if eps is None else eps))
        y = (flat * inv).reshape(B, T, H, D)
    else:
        y = _l2(tx, 1e-6 if eps is None else eps)
    if relu:
        y = torch.clamp(y, min=0.0)
    y = y * scale
    (g,) = torch.autograd.grad((y * torch.tensor(np.asarray(dy, dtype=np.float64))).sum(), (tx,))
    return g.detach().numpy()


def merge_grad(num, den, dout, gate=None, eps=1e-6):
    """Gradients of L = sum(dout . out) for the bidirectional merge out =
    num / (den + eps) * silu(gate) (SANA `fused_gdn.py` page,
    `fused_bigdn_func` / `_fused_bidi_merge_kernel`): returns dnum
    (B, T, H, V), dden (B, H, T) and, with a gate, dgate."""
    torch = _torch()
    tn, td = _t(num), _t(den)
    out = tn / (td.permute(0, 2, 1)[..., None] + eps)
    ins = [tn, td]
    if gate is not None:
        tg = _t(gate)
        out = out * (tg * torch.sigmoid(tg))
        ins.append(tg)
    grads = torch.autograd.grad((out * torch.tensor(np.asarray(dout, dtype=np.float64))).sum(), ins)
    res = {"dnum": grads[0].detach().numpy(), "dden": grads[1].detach().numpy()}
    if gate is not None:
        res["dgate"] = grads[2].detach().numpy()
    return res
