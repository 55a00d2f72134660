"""Pins for the fp64 oracle: checks against what the pages and mathematics fix,
none of which re-runs the oracle's own loop.

  * hand-worked values (tests/golden/scalar_recurrence.txt);
  * brute-force expansion of the recurrence as explicit matrix products in the
    state form `state <- state @ W + U` of the SANA `fused_cam_gdn.py` page
    (`_torch_cam_scan_single_chunk`), T <= 8;
  * closed forms: beta = 0 and g = 0 leave the state unchanged; full reset;
    a single token; exact key-value retrieval with orthonormal keys;
    mutually orthogonal keys turn the delta rule into gated linear attention
    (forward, reverse, per-key gate, denominator), computed as a masked
    matrix product;
  * invariants: split/resume equivalence (SANA `fused_cam_gdn.py` page,
    `_cam_scan_kernel` init/final state contract), reverse == flip-and-shift
    (same page, `_torch_cam_scan_reference`), varlen packing == separate
    sequences.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "scalar_recurrence.txt")


def _golden():
    d = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, vals = line.split(":", 1)
        d[key.strip()] = np.array([float(x) for x in vals.split()])
    return d


def _one(x):
    """(T, ...) single-sequence single-head arrays -> (1, T, 1, ...)."""
    return x[None, :, None]


def _run1(q, k, v, beta, g=None, gk=None, h0=None, reverse=False):
    out, hf = oracle.scan(_one(q), _one(k), _one(v), _one(beta),
                          g=None if g is None else _one(g),
                          gk=None if gk is None else _one(gk),
                          h0=None if h0 is None else h0[None, None],
                          reverse=reverse, threads=1)
    return out[0, :, 0], hf[0, 0]


# ----------------------------------------------------------------- golden ---

def test_golden_scalar_cases():
    G = _golden()
    for case, K in (("A", 1), ("C", 1), ("D", 2)):
        T = len(G[f"{case}.v"])
        q = G[f"{case}.q"].reshape(T, K)
        k = G[f"{case}.k"].reshape(T, K)
        v = G[f"{case}.v"].reshape(T, 1)
        beta = G[f"{case}.beta"]
        h0 = G[f"{case}.h0"].reshape(K, 1)
        dec = G[f"{case}.decay"]
        if dec.size == T:
            out, hf = _run1(q, k, v, beta, g=np.log(dec), h0=h0)
        else:
            out, hf = _run1(q, k, v, beta, gk=np.log(dec.reshape(T, K)), h0=h0)
        np.testing.assert_allclose(out[:, 0], G[f"{case}.out"], rtol=1e-14, atol=1e-14)
        np.testing.assert_allclose(hf[:, 0], G[f"{case}.h_final"], rtol=1e-14, atol=1e-14)
    T = 3
    out, _ = _run1(G["A.q"].reshape(T, 1), G["A.k"].reshape(T, 1),
                   G["A.v"].reshape(T, 1), G["A.beta"], g=np.log(G["A.decay"]),
                   reverse=True)
    np.testing.assert_allclose(out[:, 0], G["A.rev_out"], rtol=1e-14, atol=1e-14)


def test_golden_prep():
    G = _golden()
    y = oracle.l2norm(G["P.l2_in"][None], eps=0.0)
    np.testing.assert_allclose(y[0], G["P.l2_out"], rtol=1e-15)
    x = G["P.rms_in"].reshape(1, 1, 2, 2)
    y, inv = oracle.rmsnorm_channels(x, eps=0.0, relu=True, scale=2.0)
    np.testing.assert_allclose(inv.ravel(), G["P.rms_inv"], rtol=1e-15)
    np.testing.assert_allclose(y.ravel(), G["P.rms_out"], rtol=1e-15, atol=0)


# ------------------------------------------------------------ brute force ---

def _brute(q, k, v, beta, g=None, gk=None, h0=None):
    """M = S^T (V x K). Each token's map is M <- M W_t + U_t with
    W_t = D_t (I - beta_t k_t k_t^T), U_t = beta_t v_t k_t^T, D_t the decay.
    M_t is expanded as M_0 W_1..W_t + sum_s U_s W_{s+1}..W_t with every
    product formed explicitly."""
    T, K = k.shape
    V = v.shape[1]
    I = np.eye(K)
    W, U = [], []
    for t in range(T):
        D = np.diag(np.exp(gk[t])) if gk is not None else np.exp(g[t]) * I
        W.append(D @ (I - beta[t] * np.outer(k[t], k[t])))
        U.append(beta[t] * np.outer(v[t], k[t]))

    def chain(a, b):  # W_a W_{a+1} ... W_b  (identity if a > b)
        P = I.copy()
        for i in range(a, b + 1):
            P = P @ W[i]
        return P

    M0 = np.zeros((V, K)) if h0 is None else h0.T
    outs = []
    M = M0
    for t in range(T):
        M = M0 @ chain(0, t)
        for s in range(t + 1):
            M = M + U[s] @ chain(s + 1, t)
        outs.append(M @ q[t])
    return np.array(outs), M.T


@pytest.mark.parametrize("T,K,V,perkey", [(1, 3, 2, False), (5, 4, 3, False),
                                          (8, 3, 5, False), (7, 4, 2, True),
                                          (8, 6, 6, True)])
def test_brute_force_expansion(T, K, V, perkey):
    rng = np.random.default_rng(100 + T * 10 + K)
    q, k = rng.standard_normal((T, K)), rng.standard_normal((T, K)) * 0.6
    v = rng.standard_normal((T, V))
    beta = rng.uniform(0.1, 1.0, T)
    h0 = rng.standard_normal((K, V))
    if perkey:
        gk = -rng.uniform(0.0, 1.0, (T, K))
        got = _run1(q, k, v, beta, gk=gk, h0=h0)
        ref = _brute(q, k, v, beta, gk=gk, h0=h0)
    else:
        g = -rng.uniform(0.0, 1.0, T)
        got = _run1(q, k, v, beta, g=g, h0=h0)
        ref = _brute(q, k, v, beta, g=g, h0=h0)
    np.testing.assert_allclose(got[0], ref[0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(got[1], ref[1], rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ closed forms ---

def test_beta0_g0_state_unchanged():
    rng = np.random.default_rng(1)
    T, K, V = 13, 5, 4
    q, k, v = rng.standard_normal((T, K)), rng.standard_normal((T, K)), rng.standard_normal((T, V))
    h0 = rng.standard_normal((K, V))
    out, hf = _run1(q, k, v, np.zeros(T), g=np.zeros(T), h0=h0)
    assert np.array_equal(hf, h0)
    np.testing.assert_allclose(out, q @ h0, rtol=1e-14, atol=1e-14)


def test_full_reset():
    """g = -inf: exp(g) = 0 wipes the state before each write, so
    o_t = beta_t (q_t . k_t) v_t whatever h0 was."""
    rng = np.random.default_rng(2)
    T, K, V = 9, 4, 3
    q, k, v = rng.standard_normal((T, K)), rng.standard_normal((T, K)), rng.standard_normal((T, V))
    beta = rng.uniform(0, 1, T)
    out, hf = _run1(q, k, v, beta, g=np.full(T, -np.inf), h0=rng.standard_normal((K, V)))
    ref = (beta * np.sum(q * k, axis=1))[:, None] * v
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(hf, beta[-1] * np.outer(k[-1], v[-1]), rtol=1e-13)


def test_single_token_closed_form():
    """T = 1: S = a h0 + beta k (v - a h0^T k)^T, o = S^T q, with a = e^g."""
    rng = np.random.default_rng(3)
    K, V = 6, 5
    q, k, v = rng.standard_normal((1, K)), rng.standard_normal((1, K)), rng.standard_normal((1, V))
    h0 = rng.standard_normal((K, V))
    b, g = np.array([0.7]), np.array([-0.4])
    a = np.exp(g[0])
    S = a * h0 + b[0] * np.outer(k[0], v[0] - a * h0.T @ k[0])
    out, hf = _run1(q, k, v, b, g=g, h0=h0)
    np.testing.assert_allclose(hf, S, rtol=1e-13)
    np.testing.assert_allclose(out[0], S.T @ q[0], rtol=1e-13)


def test_orthonormal_key_value_retrieval():
    """beta = 1, g = 0, orthonormal keys: after writing (k_i, v_i) the memory
    returns v_i for k_i exactly, and later orthogonal writes leave it."""
    rng = np.random.default_rng(4)
    T, K, V = 6, 8, 5
    Qm, _ = np.linalg.qr(rng.standard_normal((K, K)))
    k = Qm[:, :T].T
    v = rng.standard_normal((T, V))
    idx = np.array([rng.integers(0, t + 1) for t in range(T)])  # i(t) <= t
    q = k[idx]
    out, hf = _run1(q, k, v, np.ones(T), g=np.zeros(T))
    np.testing.assert_allclose(out, v[idx], atol=1e-13)
    np.testing.assert_allclose(k @ hf, v, atol=1e-13)


def _orth_keys(rng, T, K, scale=True):
    Qm, _ = np.linalg.qr(rng.standard_normal((K, K)))
    k = Qm[:, :T].T
    if scale:
        k = k * rng.uniform(0.5, 2.0, (T, 1))
    return k


def test_orthogonal_keys_is_gated_linear_attention():
    """Mutually orthogonal keys and h0 = 0: the prediction S^T k_t is always 0,
    so delta_t = beta_t v_t and
      o_t = sum_{j<=t} exp(G_t - G_j) beta_j (q_t . k_j) v_j,  G = cumsum g."""
    rng = np.random.default_rng(5)
    T, K, V = 10, 12, 4
    k = _orth_keys(rng, T, K)
    q, v = rng.standard_normal((T, K)), rng.standard_normal((T, V))
    beta, g = rng.uniform(0.1, 1, T), -rng.uniform(0, 0.7, T)
    G = np.cumsum(g)
    L = np.tril(np.exp(G[:, None] - G[None, :]))
    ref = ((q @ k.T) * L * beta[None, :]) @ v
    out, _ = _run1(q, k, v, beta, g=g)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    # the denominator: the same with v = 1
    d = oracle.den(_one(q), _one(k), _one(beta), g=_one(g))[0, 0]
    np.testing.assert_allclose(d, ((q @ k.T) * L * beta[None, :]).sum(1), rtol=1e-12, atol=1e-12)


def test_orthogonal_keys_reverse_closed_form():
    """Reverse scan, orthogonal keys: token p reads tokens j > p,
      o_p = sum_{j>p} beta_j (q_p . k_j) v_j exp(g_{p+1} + ... + g_{j-1}),
    i.e. no self term and a token's own gate does not decay its own write."""
    rng = np.random.default_rng(6)
    T, K, V = 9, 10, 3
    k = _orth_keys(rng, T, K)
    q, v = rng.standard_normal((T, K)), rng.standard_normal((T, V))
    beta, g = rng.uniform(0.1, 1, T), -rng.uniform(0, 0.7, T)
    ref = np.zeros((T, V))
    for p in range(T):
        for j in range(p + 1, T):
            ref[p] += beta[j] * (q[p] @ k[j]) * v[j] * np.exp(g[p + 1:j].sum())
    out, _ = _run1(q, k, v, beta, g=g, reverse=True)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_disjoint_keys_per_key_gate_closed_form():
    """Keys on distinct coordinate axes stay orthogonal under any per-key
    decay, so o_t = sum_{j<=t} beta_j (sum_d q_td k_jd e^{Gk_td - Gk_jd}) v_j."""
    rng = np.random.default_rng(7)
    T, K, V = 7, 9, 4
    perm = rng.permutation(K)[:T]
    k = np.zeros((T, K))
    k[np.arange(T), perm] = rng.uniform(0.5, 2.0, T)
    q, v = rng.standard_normal((T, K)), rng.standard_normal((T, V))
    beta, gk = rng.uniform(0.1, 1, T), -rng.uniform(0, 0.7, (T, K))
    Gk = np.cumsum(gk, axis=0)
    ref = np.zeros((T, V))
    for t in range(T):
        for j in range(t + 1):
            a = np.sum(q[t] * k[j] * np.exp(Gk[t] - Gk[j]))
            ref[t] += beta[j] * a * v[j]
    out, _ = _run1(q, k, v, beta, gk=gk)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


# -------------------------------------------------------------- invariants ---

def test_split_resume_equivalence():
    rng = np.random.default_rng(8)
    T, K, V, t0 = 40, 6, 5, 17
    q, k, v = rng.standard_normal((T, K)), rng.standard_normal((T, K)) * 0.4, rng.standard_normal((T, V))
    beta, gk = rng.uniform(0, 1, T), -rng.uniform(0, 0.3, (T, K))
    full_o, full_h = _run1(q, k, v, beta, gk=gk)
    pre_o, pre_h = _run1(q[:t0], k[:t0], v[:t0], beta[:t0], gk=gk[:t0])
    suf_o, suf_h = _run1(q[t0:], k[t0:], v[t0:], beta[t0:], gk=gk[t0:], h0=pre_h)
    assert np.array_equal(full_o, np.concatenate([pre_o, suf_o]))
    assert np.array_equal(full_h, suf_h)


def _flip_shift(x, pad):
    y = np.flip(x, 0)
    return np.concatenate([np.full((1,) + x.shape[1:], pad), y[:-1]], 0)


def test_reverse_equals_flip_and_shift():
    """Reverse scan == forward scan on q flipped, k, v, beta flipped and
    shifted (pad 0), gate flipped and shifted (pad log 1 = 0), flipped back."""
    rng = np.random.default_rng(9)
    T, K, V = 23, 5, 4
    q, k, v = rng.standard_normal((T, K)), rng.standard_normal((T, K)) * 0.5, rng.standard_normal((T, V))
    beta, g = rng.uniform(0, 1, T), -rng.uniform(0, 0.5, T)
    rev, _ = _run1(q, k, v, beta, g=g, reverse=True)
    fwd, _ = _run1(np.flip(q, 0), _flip_shift(k, 0.0), _flip_shift(v, 0.0),
                   _flip_shift(beta, 0.0), g=_flip_shift(g, 0.0))
    np.testing.assert_allclose(rev, np.flip(fwd, 0), rtol=1e-13, atol=1e-13)
    assert np.all(rev[-1] == 0.0)


def test_varlen_packing_equals_separate_sequences():
    rng = np.random.default_rng(10)
    lens = [5, 1, 12, 0, 7]
    T, H, K, V = sum(lens), 3, 4, 3
    q, k = rng.standard_normal((1, T, H, K)), rng.standard_normal((1, T, H, K)) * 0.5
    v = rng.standard_normal((1, T, H, V))
    beta, g = rng.uniform(0, 1, (1, T, H)), -rng.uniform(0, 0.5, (1, T, H))
    h0 = rng.standard_normal((len(lens), H, K, V))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    out, hf = oracle.scan(q, k, v, beta, g=g, h0=h0, cu_seqlens=cu)
    for s in range(len(lens)):
        a, b = cu[s], cu[s + 1]
        o_s, h_s = oracle.scan(q[:, a:b], k[:, a:b], v[:, a:b], beta[:, a:b],
                               g=g[:, a:b], h0=h0[s:s + 1])
        assert np.array_equal(out[:, a:b], o_s)
        assert np.array_equal(hf[s], h_s[0])
    assert np.array_equal(hf[3], h0[3])  # empty sequence passes h0 through


def test_threads_do_not_change_results():
    rng = np.random.default_rng(11)
    B, T, H, K, V = 2, 30, 5, 4, 3
    args = [rng.standard_normal((B, T, H, K)), rng.standard_normal((B, T, H, K)),
            rng.standard_normal((B, T, H, V)), rng.uniform(0, 1, (B, T, H))]
    g = -rng.uniform(0, 1, (B, T, H))
    o1, h1 = oracle.scan(*args, g=g, threads=1)
    o7, h7 = oracle.scan(*args, g=g, threads=7)
    assert np.array_equal(o1, o7) and np.array_equal(h1, h7)


# -------------------------------------------------------------------- prep ---

def test_l2norm_invariants():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((50, 64)) * rng.uniform(0.1, 10, (50, 1))
    y = oracle.l2norm(x, eps=1e-6)
    n2 = (x * x).sum(1)
    # y = c x with c > 0, and |y|^2 = n2 / (n2 + eps)
    c = (y * x).sum(1) / n2
    np.testing.assert_allclose(y, c[:, None] * x, rtol=1e-14)
    np.testing.assert_allclose((y * y).sum(1), n2 / (n2 + 1e-6), rtol=1e-13)
    # scale invariance when eps = 0
    np.testing.assert_allclose(oracle.l2norm(3.5 * x, eps=0.0), oracle.l2norm(x, eps=0.0), rtol=1e-14)


def test_rmsnorm_channels_invariants():
    rng = np.random.default_rng(13)
    x = rng.standard_normal((2, 7, 4, 6)) * rng.uniform(0.2, 5, (2, 7, 1, 1))
    y, inv = oracle.rmsnorm_channels(x, eps=0.0)
    np.testing.assert_allclose((y ** 2).mean(axis=(2, 3)), 1.0, rtol=1e-13)
    yr, _ = oracle.rmsnorm_channels(x, eps=0.0, relu=True, scale=0.25)
    np.testing.assert_allclose(yr, 0.25 * np.maximum(y, 0.0), rtol=1e-15)
    # channels of other heads matter: the norm is over all H*D channels
    x2 = x.copy()
    x2[:, :, 1] *= 3.0
    y2, _ = oracle.rmsnorm_channels(x2, eps=0.0)
    assert not np.allclose(y2[:, :, 0], y[:, :, 0])


def test_merge_closed_form():
    # out = num / (den + eps) * silu(gate) (SANA `fused_gdn.py` page,
    # `fused_bigdn_func` and `_fused_bidi_merge_kernel`): worked values
    num = np.array([3.0, -3.0, 6.0, 0.0]).reshape(1, 1, 1, 4)
    den = np.array([1.0]).reshape(1, 1, 1)
    np.testing.assert_allclose(oracle.merge(num, den, eps=0.5), [[[[2.0, -2.0, 4.0, 0.0]]]],
                               rtol=0, atol=1e-15)
    # silu(ln 3) = ln 3 / (1 + 1/3) = 0.75 ln 3; silu(0) = 0; silu(-ln 3) = -0.25 ln 3
    gate = np.array([np.log(3.0), np.log(3.0), 0.0, -np.log(3.0)]).reshape(1, 1, 1, 4)
    want = np.array([2.0 * 0.75, -2.0 * 0.75, 0.0, 0.0]) * np.log(3.0)
    np.testing.assert_allclose(oracle.merge(num, den, gate=gate, eps=0.5)[0, 0, 0], want,
                               rtol=1e-15, atol=1e-15)
    # den is indexed (B, H, T): a transposed den must move to the right rows
    num2 = np.ones((1, 2, 3, 4))
    den2 = np.arange(6, dtype=np.float64).reshape(1, 3, 2)  # (B, H, T)
    got = oracle.merge(num2, den2, eps=1.0)
    for t in range(2):
        for h in range(3):
            np.testing.assert_allclose(got[0, t, h], 1.0 / (den2[0, h, t] + 1.0), rtol=1e-15)


@pytest.mark.parametrize("b", [1, 5, 10])
def test_reverse_reset_splits_the_sequence(b):
    # Chunk-causal backward direction (SANA `fused_gdn.py` page: decay_bwd
    # zeroed at boundary frames): with the log-gate of token b at -inf, the
    # reverse scan of the whole sequence equals, for positions p < b, the
    # reverse scan of tokens 0..b alone and, for p >= b, that of tokens b..T-1
    # alone (position p reads tokens p+1.. ; token b's decay wipes what came
    # after it before its own update lands).
    rng = np.random.default_rng(7)
    T, K, V = 12, 4, 3
    q, k = rng.normal(size=(T, K)), rng.normal(size=(T, K))
    v, beta = rng.normal(size=(T, V)), rng.uniform(0.1, 0.9, size=T)
    g = np.log(rng.uniform(0.5, 0.99, size=T))
    g_reset = g.copy()
    g_reset[b] = -np.inf
    full, _ = oracle.scan(*map(_one, (q, k, v, beta, g_reset)), reverse=True)
    pre, _ = oracle.scan(*map(_one, (q[:b + 1], k[:b + 1], v[:b + 1], beta[:b + 1], g[:b + 1])),
                         reverse=True)
    suf, _ = oracle.scan(*map(_one, (q[b:], k[b:], v[b:], beta[b:], g[b:])), reverse=True)
    np.testing.assert_allclose(full[0, :b, 0], pre[0, :b, 0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(full[0, b:, 0], suf[0, :, 0], rtol=1e-12, atol=1e-12)
    # without the reset the early positions see the later tokens
    plain, _ = oracle.scan(*map(_one, (q, k, v, beta, g)), reverse=True)
    assert np.abs(plain[0, :b, 0] - pre[0, :b, 0]).max() > 1e-3


# ------------------------------------------------------------ frame-causal ---

def _frame_rand(seed, B, F, S, H, K, V):
    rng = np.random.default_rng(seed)
    T = F * S
    q, k = rng.normal(size=(B, T, H, K)), rng.normal(size=(B, T, H, K)) * 0.5
    v, beta = rng.normal(size=(B, T, H, V)), rng.uniform(0.1, 0.9, (B, T, H))
    gf = np.log(rng.uniform(0.5, 0.99, (B, F, H)))
    return q, k, v, beta, gf


@pytest.mark.parametrize("reverse", [False, True])
def test_frame_of_one_token_is_the_token_rule(reverse):
    # one token per frame: the SANA kernels' frame rule is exactly the token
    # rule, with the per-frame decay as the per-token gate
    q, k, v, beta, gf = _frame_rand(21, 2, 9, 1, 3, 4, 3)
    h0 = None if reverse else np.random.default_rng(22).normal(size=(2, 3, 4, 3))
    of, hf = oracle.frame_scan(q, k, v, beta, gf, 1, h0=h0, reverse=reverse)
    ot, ht = oracle.scan(q, k, v, beta, g=gf, h0=h0, reverse=reverse)
    np.testing.assert_allclose(of, ot, rtol=0, atol=1e-14)
    np.testing.assert_allclose(hf, ht, rtol=0, atol=1e-14)


def test_frame_rule_matrix_form():
    # per frame, as matrix products (SANA `fused_gdn.py` page, Pass 1 with a
    # fixed state_prev): S_pre = e^{g_f} S; S = S_pre + K^T diag(beta)(V - K S_pre);
    # then O = Q S for the frame's tokens
    B, F, S, H, K, V = 1, 4, 5, 2, 3, 4
    q, k, v, beta, gf = _frame_rand(23, B, F, S, H, K, V)
    h0 = np.random.default_rng(24).normal(size=(B, H, K, V))
    out, hf = oracle.frame_scan(q, k, v, beta, gf, S, h0=h0)
    for h in range(H):
        St = h0[0, h].copy()
        for f in range(F):
            rows = slice(f * S, (f + 1) * S)
            Kf, Vf, Qf = k[0, rows, h], v[0, rows, h], q[0, rows, h]
            Spre = np.exp(gf[0, f, h]) * St
            St = Spre + Kf.T @ (beta[0, rows, h][:, None] * (Vf - Kf @ Spre))
            np.testing.assert_allclose(out[0, rows, h], Qf @ St, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(hf[0, h], St, rtol=1e-12, atol=1e-12)


def test_frame_reverse_is_frame_flip_and_shift():
    # reverse at frame granularity (`_fused_gdn_kernel` REVERSE: q_frame =
    # F-1-i, kv_frame = F-i, no update and decay 1 at i = 0) == the forward
    # frame rule on frames taken in reverse order, k / v / beta / decay moved
    # one frame later (pad 0, decay pad 0 = log 1), outputs put back
    B, F, S, H, K, V = 2, 5, 3, 2, 4, 3
    q, k, v, beta, gf = _frame_rand(25, B, F, S, H, K, V)
    rev, _ = oracle.frame_scan(q, k, v, beta, gf, S, reverse=True)

    def frames(x):
        return x.reshape(x.shape[0], F, S, *x.shape[2:])

    def flip_shift(x, pad):
        xf = frames(x)[:, ::-1]
        y = np.full_like(xf, pad)
        y[:, 1:] = xf[:, :-1]
        return y.reshape(x.shape)
    qf = frames(q)[:, ::-1].reshape(q.shape)
    g2 = np.zeros_like(gf)
    g2[:, 1:] = gf[:, ::-1][:, :-1]
    fwd, _ = oracle.frame_scan(qf, flip_shift(k, 0.0), flip_shift(v, 0.0), flip_shift(beta, 0.0),
                               g2, S)
    back = frames(fwd)[:, ::-1].reshape(fwd.shape)
    np.testing.assert_allclose(rev, back, rtol=1e-13, atol=1e-13)
    assert np.all(frames(rev)[:, -1] == 0.0)


# ------------------------------------------- segment summaries (state_ext, M) ---
# hyper-parallel coverage_diff page, `kda_state_summary_forward_from_prepared`:
# a piece's final state is transition . h_in + state_ext.

def test_summary_one_token_segments_closed_form():
    """segment_len = 1: M_t = (I - beta_t k_t k_t^T) e^{g_t} and
    E_t = beta_t k_t v_t^T, written out from the update rule (decay, predict,
    correct); per-key gate: M_t = (I - beta k k^T) diag(e^{gk_t})."""
    rng = np.random.default_rng(31)
    T, K, V = 3, 5, 4
    k, v = rng.standard_normal((T, K)), rng.standard_normal((T, V))
    beta, g = rng.uniform(0.1, 1, T), -rng.uniform(0, 1, T)
    gk = -rng.uniform(0, 1, (T, K))
    ext, tr = oracle.state_summary(_one(k), _one(v), _one(beta), 1, g=_one(g), threads=1)
    _, trk = oracle.state_summary(_one(k), _one(v), _one(beta), 1, gk=_one(gk), threads=1)
    for t in range(T):
        P = np.eye(K) - beta[t] * np.outer(k[t], k[t])
        np.testing.assert_allclose(tr[t, 0, 0], P * np.exp(g[t]), rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(ext[t, 0, 0], beta[t] * np.outer(k[t], v[t]), rtol=1e-13)
        np.testing.assert_allclose(trk[t, 0, 0], P @ np.diag(np.exp(gk[t])), rtol=1e-13, atol=1e-15)


def test_summary_beta0_is_pure_decay():
    """beta = 0: nothing is written; M = e^{sum g} I (diag(e^{sum gk})), E = 0."""
    rng = np.random.default_rng(32)
    T, K, V = 7, 4, 3
    k, v = rng.standard_normal((T, K)), rng.standard_normal((T, V))
    g, gk = -rng.uniform(0, 1, T), -rng.uniform(0, 1, (T, K))
    ext, tr = oracle.state_summary(_one(k), _one(v), _one(np.zeros(T)), T, g=_one(g), threads=1)
    np.testing.assert_array_equal(ext, 0.0)
    np.testing.assert_allclose(tr[0, 0, 0], np.exp(g.sum()) * np.eye(K), rtol=1e-13, atol=1e-16)
    _, trk = oracle.state_summary(_one(k), _one(v), _one(np.zeros(T)), T, gk=_one(gk), threads=1)
    np.testing.assert_allclose(trk[0, 0, 0], np.diag(np.exp(gk.sum(0))), rtol=1e-13, atol=1e-16)


def test_summary_composes_over_adjacent_segments():
    """Two halves compose into the whole: M = M2 M1, E = M2 E1 + E2 (a
    transposed or reversed product fails)."""
    rng = np.random.default_rng(33)
    T, K, V = 12, 5, 3
    k, v = rng.standard_normal((T, K)) / np.sqrt(K), rng.standard_normal((T, V))
    beta, g = rng.uniform(0, 1, T), -rng.uniform(0, 0.5, T)
    half, whole = (oracle.state_summary(_one(k), _one(v), _one(beta), L, g=_one(g), threads=1)
                   for L in (6, 12))
    (E1, E2), (M1, M2) = half[0][:, 0, 0], half[1][:, 0, 0]
    np.testing.assert_allclose(whole[1][0, 0, 0], M2 @ M1, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(whole[0][0, 0, 0], M2 @ E1 + E2, rtol=1e-12, atol=1e-14)


def test_summary_reproduces_scan_from_any_state():
    """Ragged last segment: applying the summaries segment by segment from a
    random h0 gives the scan's final state from h0."""
    rng = np.random.default_rng(34)
    B, T, H, K, V = 2, 11, 2, 4, 3
    k, v = rng.standard_normal((B, T, H, K)) / 2, rng.standard_normal((B, T, H, V))
    beta, g = rng.uniform(0, 1, (B, T, H)), -rng.uniform(0, 0.5, (B, T, H))
    h0 = rng.standard_normal((B, H, K, V))
    ext, tr = oracle.state_summary(k, v, beta, 4, g=g, threads=1)
    assert ext.shape == (3, B, H, K, V) and tr.shape == (3, B, H, K, K)
    h = h0.copy()
    for s in range(3):
        h = tr[s] @ h + ext[s]
    _, hf = oracle.scan(k, k, v, beta, g=g, h0=h0, threads=1)
    np.testing.assert_allclose(h, hf, rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------- gradients ---
# oracle/backward.py differentiates the plain token loop with autograd; it is
# pinned to central finite differences of the C forward oracle (a separate
# implementation) and to the beta = 0 closed form.

def _fd_case(seed, B, T, H, K, V):
    rng = np.random.default_rng(seed)
    x = dict(q=rng.standard_normal((B, T, H, K)), k=rng.standard_normal((B, T, H, K)) / np.sqrt(K),
             v=rng.standard_normal((B, T, H, V)), beta=rng.uniform(0.2, 0.9, (B, T, H)),
             g=-rng.uniform(0.05, 0.6, (B, T, H)), h0=rng.standard_normal((B, H, K, V)))
    return x, rng.standard_normal((B, T, H, V)), rng.standard_normal((B, H, K, V))


def _loss_c(x, do, dhf, reverse, l2norm):
    """L = sum(do o) + sum(dh_final h_final) through the C forward oracle."""
    q, k = (oracle.l2norm(x["q"]), oracle.l2norm(x["k"])) if l2norm else (x["q"], x["k"])
    o, hf = oracle.scan(q, k, x["v"], x["beta"], g=x["g"], h0=None if reverse else x["h0"],
                        reverse=reverse, threads=1)
    return float(np.sum(do * o) + (0.0 if reverse else np.sum(dhf * hf)))


@pytest.mark.parametrize("reverse,l2norm", [(False, False), (False, True), (True, False)])
def test_gradients_match_central_differences(reverse, l2norm):
    from oracle import backward
    x, do, dhf = _fd_case(41 + 2 * reverse + l2norm, 1, 5, 2, 3, 2)
    res = backward.scan_grad(x["q"], x["k"], x["v"], x["beta"], x["g"], do,
                             h0=None if reverse else x["h0"], dh_final=None if reverse else dhf,
                             reverse=reverse, l2norm=l2norm)
    eps = 1e-6
    for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("beta", "dbeta"), ("g", "dg"),
                        ("h0", "dh0")):
        if reverse and name == "h0":
            continue
        fd = np.zeros_like(x[name])
        for ix in np.ndindex(x[name].shape):
            xp = {n: a.copy() for n, a in x.items()}
            xm = {n: a.copy() for n, a in x.items()}
            xp[name][ix] += eps
            xm[name][ix] -= eps
            fd[ix] = (_loss_c(xp, do, dhf, reverse, l2norm) - _loss_c(xm, do, dhf, reverse, l2norm)) / (2 * eps)
        np.testing.assert_allclose(res[gname], fd, rtol=1e-6, atol=1e-8, err_msg=gname)


def test_gradients_varlen_match_central_differences():
    """Packed sequences (one empty, one of one token), each from its own h0:
    the autograd gradients against central differences of the C oracle's
    variable-length forward, on every input coordinate."""
    from oracle import backward
    lens = [3, 0, 1, 4]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, H, K, V, n = int(cu[-1]), 2, 3, 2, len(lens)
    rng = np.random.default_rng(48)
    x = dict(q=rng.standard_normal((1, T, H, K)), k=rng.standard_normal((1, T, H, K)) / np.sqrt(K),
             v=rng.standard_normal((1, T, H, V)), beta=rng.uniform(0.2, 0.9, (1, T, H)),
             g=-rng.uniform(0.05, 0.6, (1, T, H)), h0=rng.standard_normal((n, H, K, V)))
    do, dhf = rng.standard_normal((1, T, H, V)), rng.standard_normal((n, H, K, V))

    def loss(y):
        q, k = oracle.l2norm(y["q"]), oracle.l2norm(y["k"])
        o, hf = oracle.scan(q, k, y["v"], y["beta"], g=y["g"], h0=y["h0"], cu_seqlens=cu, threads=1)
        return float(np.sum(do * o) + np.sum(dhf * hf))
    res = backward.scan_grad(x["q"], x["k"], x["v"], x["beta"], x["g"], do, h0=x["h0"],
                             dh_final=dhf, l2norm=True, cu_seqlens=cu)
    eps = 1e-6
    for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("beta", "dbeta"), ("g", "dg"),
                        ("h0", "dh0")):
        fd = np.zeros_like(x[name])
        for ix in np.ndindex(x[name].shape):
            xp = {n_: a.copy() for n_, a in x.items()}
            xm = {n_: a.copy() for n_, a in x.items()}
            xp[name][ix] += eps
            xm[name][ix] -= eps
            fd[ix] = (loss(xp) - loss(xm)) / (2 * eps)
        np.testing.assert_allclose(res[gname], fd, rtol=1e-6, atol=1e-8, err_msg=gname)
    # the empty sequence passes its final-state gradient straight through
    np.testing.assert_array_equal(res["dh0"][1], dhf[1])


def test_gradients_per_key_gate_match_central_differences():
    """Per-key gates (the state's key rows decay separately), with L2 prep,
    h0 and dh_final: autograd against central differences of the C oracle."""
    from oracle import backward
    x, do, dhf = _fd_case(49, 1, 5, 2, 3, 2)
    gk = -np.random.default_rng(50).uniform(0.05, 0.8, (1, 5, 2, 3))

    def loss(y, gk_):
        q, k = oracle.l2norm(y["q"]), oracle.l2norm(y["k"])
        o, hf = oracle.scan(q, k, y["v"], y["beta"], gk=gk_, h0=y["h0"], threads=1)
        return float(np.sum(do * o) + np.sum(dhf * hf))
    res = backward.scan_grad(x["q"], x["k"], x["v"], x["beta"], None, do, h0=x["h0"],
                             dh_final=dhf, l2norm=True, gk=gk)
    eps = 1e-6
    fd = np.zeros_like(gk)
    for ix in np.ndindex(gk.shape):
        gp, gm = gk.copy(), gk.copy()
        gp[ix] += eps
        gm[ix] -= eps
        fd[ix] = (loss(x, gp) - loss(x, gm)) / (2 * eps)
    np.testing.assert_allclose(res["dg"], fd, rtol=1e-6, atol=1e-8, err_msg="dgk")
    for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("beta", "dbeta"), ("h0", "dh0")):
        fd = np.zeros_like(x[name])
        for ix in np.ndindex(x[name].shape):
            xp = {n_: a.copy() for n_, a in x.items()}
            xm = {n_: a.copy() for n_, a in x.items()}
            xp[name][ix] += eps
            xm[name][ix] -= eps
            fd[ix] = (loss(xp, gk) - loss(xm, gk)) / (2 * eps)
        np.testing.assert_allclose(res[gname], fd, rtol=1e-6, atol=1e-8, err_msg=gname)


@pytest.mark.parametrize("direction", [0, 1, 2])
def test_frame_gradients_match_central_differences(direction):
    """Frame-causal rule (frames of 2 tokens) with the denominator's upstream
    gradient, and h0 / dh_final in the causal direction: autograd of the
    frame loop against central differences of the C oracle's frame scan."""
    from oracle import backward
    rng = np.random.default_rng(60 + direction)
    B, F, S, H, K, V = 1, 3, 2, 2, 3, 2
    T = F * S
    x = dict(q=rng.standard_normal((B, T, H, K)), k=rng.standard_normal((B, T, H, K)) / 2,
             v=rng.standard_normal((B, T, H, V)), beta=rng.uniform(0.2, 0.9, (B, T, H)),
             g=-rng.uniform(0.1, 0.6, (B, F, H)), h0=rng.standard_normal((B, H, K, V)))
    do, dden = rng.standard_normal((B, T, H, V)), rng.standard_normal((B, H, T))
    dhf = rng.standard_normal((B, H, K, V))
    state = direction == 0

    def loss(y):
        tot = 0.0
        for rev in ([False], [True], [False, True])[direction]:
            o, hf = oracle.frame_scan(y["q"], y["k"], y["v"], y["beta"], y["g"], S,
                                      h0=y["h0"] if state else None, reverse=rev, threads=1)
            d = oracle.frame_den(y["q"], y["k"], y["beta"], y["g"], S, reverse=rev, threads=1)
            tot += float(np.sum(do * o) + np.sum(dden * d))
            if state:
                tot += float(np.sum(dhf * hf))
        return tot
    res = backward.frame_grad(x["q"], x["k"], x["v"], x["beta"], x["g"], S, do, dden=dden,
                              h0=x["h0"] if state else None, dh_final=dhf if state else None,
                              direction=direction)
    eps = 1e-6
    names = [("q", "dq"), ("k", "dk"), ("v", "dv"), ("beta", "dbeta"), ("g", "dg_frame")]
    if state:
        names.append(("h0", "dh0"))
    for name, gname in names:
        fd = np.zeros_like(x[name])
        for ix in np.ndindex(x[name].shape):
            xp = {n_: a.copy() for n_, a in x.items()}
            xm = {n_: a.copy() for n_, a in x.items()}
            xp[name][ix] += eps
            xm[name][ix] -= eps
            fd[ix] = (loss(xp) - loss(xm)) / (2 * eps)
        np.testing.assert_allclose(res[gname], fd, rtol=1e-6, atol=1e-8, err_msg=gname)
    if direction == 1:  # the reverse scan never reads frame 0's keys and values
        np.testing.assert_array_equal(res["dv"][:, :S], 0.0)
        np.testing.assert_array_equal(res["dg_frame"][:, 0], 0.0)


@pytest.mark.parametrize("rms,relu,scale", [(False, False, 1.0), (False, True, 0.5), (True, True, 0.3),
                                             (True, False, 1.0)])
def test_prep_gradients_match_central_differences(rms, relu, scale):
    """The q/k preparation's gradient against central differences of the C
    oracle's L2 and full-channel RMS normalisations."""
    from oracle import backward
    rng = np.random.default_rng(70 + 2 * rms + relu)
    x = rng.standard_normal((1, 3, 2, 4))
    dy = rng.standard_normal(x.shape)

    def f(z):
        if rms:
            y, _ = oracle.rmsnorm_channels(z, 1e-5, relu=relu, scale=scale)
        else:
            y = oracle.l2norm(z)
            y = (np.maximum(y, 0.0) if relu else y) * scale
        return float(np.sum(y * dy))
    got = backward.prep_grad(x, dy, rms=rms, relu=relu, scale=scale)
    fd = np.zeros_like(x)
    for ix in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[ix] += 1e-6
        xm[ix] -= 1e-6
        fd[ix] = (f(xp) - f(xm)) / 2e-6
    np.testing.assert_allclose(got, fd, rtol=1e-6, atol=1e-8)


@pytest.mark.parametrize("with_gate", [False, True])
def test_merge_gradients_match_central_differences(with_gate):
    """The merge's gradients against central differences of oracle.merge."""
    from oracle import backward
    rng = np.random.default_rng(90 + with_gate)
    num = rng.standard_normal((1, 3, 2, 4))
    den = rng.uniform(0.2, 2.0, (1, 2, 3))
    gate = rng.standard_normal(num.shape) * 2 if with_gate else None
    dout = rng.standard_normal(num.shape)
    res = backward.merge_grad(num, den, dout, gate=gate, eps=1e-3)
    x = {"num": num, "den": den}
    if with_gate:
        x["gate"] = gate

    def f(y):
        return float(np.sum(dout * oracle.merge(y["num"], y["den"], gate=y.get("gate"), eps=1e-3)))
    for name in x:
        fd = np.zeros_like(x[name])
        for ix in np.ndindex(x[name].shape):
            xp = {n_: a.copy() for n_, a in x.items()}
            xm = {n_: a.copy() for n_, a in x.items()}
            xp[name][ix] += 1e-6
            xm[name][ix] -= 1e-6
            fd[ix] = (f(xp) - f(xm)) / 2e-6
        np.testing.assert_allclose(res["d" + name], fd, rtol=1e-6, atol=1e-8, err_msg=name)


def test_gradients_beta0_closed_form():
    """beta = 0: o_t = e^{G_t} h0^T q_t and h_final = e^{G_T} h0 with G the
    running sum of g, so dq_t = e^{G_t} h0 do_t, dh0 = sum_t e^{G_t} q_t do_t^T
    + e^{G_T} dh_final, dk = dv = 0 and dg_t = sum_{s >= t} (the terms of L
    that G_s multiplies)."""
    from oracle import backward
    x, do, dhf = _fd_case(47, 1, 6, 1, 3, 2)
    q, g, h0 = x["q"][0, :, 0], x["g"][0, :, 0], x["h0"][0, 0]
    dd = do[0, :, 0]
    res = backward.scan_grad(x["q"], x["k"], x["v"], np.zeros_like(x["beta"]), x["g"], do,
                             h0=x["h0"], dh_final=dhf)
    G = np.cumsum(g)
    e = np.exp(G)
    np.testing.assert_allclose(res["dq"][0, :, 0], e[:, None] * (dd @ h0.T), rtol=1e-12)
    np.testing.assert_allclose(res["dh0"][0, 0], (e[:, None] * q).T @ dd + e[-1] * dhf[0, 0],
                               rtol=1e-12)
    np.testing.assert_array_equal(res["dk"], 0.0)
    np.testing.assert_array_equal(res["dv"], 0.0)
    terms = e * np.einsum("tk,kv,tv->t", q, h0, dd)
    terms[-1] += e[-1] * np.sum(dhf[0, 0] * h0)
    np.testing.assert_allclose(res["dg"][0, :, 0], np.cumsum(terms[::-1])[::-1], rtol=1e-12)


# ------------------------------------------ denominators and the forward glue ---
# SANA `fused_gdn.py` page, `_fused_gdn_kernel`: the z state (`z_hat`, `dz`,
# `den`) runs the same rule as the numerator with a ones value, in either
# direction (REVERSE); `fused_bigdn_func` sums both directions of num and den.

def test_orthogonal_keys_reverse_den_closed_form():
    """Reverse denominator, mutually orthogonal keys: the reverse closed form
    with v = 1,  den_p = sum_{j>p} beta_j (q_p . k_j) exp(g_{p+1} + ... + g_{j-1})."""
    rng = np.random.default_rng(31)
    T, K = 9, 11
    k = _orth_keys(rng, T, K)
    q = rng.standard_normal((T, K))
    beta, g = rng.uniform(0.1, 1, T), -rng.uniform(0, 0.7, T)
    ref = np.zeros(T)
    for p in range(T):
        for j in range(p + 1, T):
            ref[p] += beta[j] * (q[p] @ k[j]) * np.exp(g[p + 1:j].sum())
    d = oracle.den(_one(q), _one(k), _one(beta), g=_one(g), reverse=True)[0, 0]
    np.testing.assert_allclose(d, ref, rtol=1e-12, atol=1e-12)
    # the causal one differs (it includes the self term and earlier tokens)
    dc = oracle.den(_one(q), _one(k), _one(beta), g=_one(g))[0, 0]
    assert np.abs(dc - ref).max() > 1e-3



# the z state carried in and out of a call (`_fused_gdn_kernel`'s
# init_state_z and its final z): z is a K-vector with
#   z_t = e^{g_t} (I - beta_t k_t k_t^T) z_{t-1} + beta_t k_t,  den_t = q_t . z_t
# (the rule's state with a single ones column; the matrix is symmetric)

def test_den_z_state_matrix_recurrence():
    rng = np.random.default_rng(33)
    B, T, H, K = 2, 8, 3, 5
    q, k = rng.standard_normal((B, T, H, K)), rng.standard_normal((B, T, H, K)) * 0.5
    beta, g = rng.uniform(0, 1, (B, T, H)), -rng.uniform(0, 0.6, (B, T, H))
    z0 = rng.standard_normal((B, H, K))
    want = np.zeros((B, H, T))
    zf = np.zeros((B, H, K))
    for b in range(B):
        for h in range(H):
            z = z0[b, h].copy()
            for t in range(T):
                kt = k[b, t, h]
                z = np.exp(g[b, t, h]) * (np.eye(K) - beta[b, t, h] * np.outer(kt, kt)) @ z + beta[b, t, h] * kt
                want[b, h, t] = q[b, t, h] @ z
            zf[b, h] = z
    got, got_zf = oracle.den(q, k, beta, g=g, z0=z0, with_state=True)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(got_zf, zf, rtol=1e-12, atol=1e-12)


def test_den_z_state_beta_zero_closed_form():
    """beta = 0: nothing is written, z_t = exp(sum_{s<=t} gk_s) * z0
    elementwise (per-key gate), den_t = q_t . z_t."""
    rng = np.random.default_rng(34)
    T, K = 6, 4
    q = rng.standard_normal((T, K))
    gk = -rng.uniform(0, 0.5, (T, K))
    z0 = rng.standard_normal(K)
    zt = np.exp(np.cumsum(gk, axis=0)) * z0
    d, zf = oracle.den(_one(q), _one(rng.standard_normal((T, K))), _one(np.zeros(T)), gk=_one(gk),
                       z0=z0[None, None], with_state=True)
    np.testing.assert_allclose(d[0, 0], np.einsum("tk,tk->t", q, zt), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(zf[0, 0], zt[-1], rtol=1e-13, atol=1e-13)


def test_den_z_state_split_resume():
    """A stream split into two calls, the second starting from the first's
    final z, gives the unsplit denominator and final z."""
    rng = np.random.default_rng(35)
    T, K, t0 = 30, 6, 13
    q, k = rng.standard_normal((T, K)), rng.standard_normal((T, K)) * 0.4
    beta, g = rng.uniform(0, 1, T), -rng.uniform(0, 0.4, T)
    full, zf = oracle.den(_one(q), _one(k), _one(beta), g=_one(g), with_state=True)
    pre, zp = oracle.den(_one(q[:t0]), _one(k[:t0]), _one(beta[:t0]), g=_one(g[:t0]), with_state=True)
    suf, zs = oracle.den(_one(q[t0:]), _one(k[t0:]), _one(beta[t0:]), g=_one(g[t0:]), z0=zp,
                         with_state=True)
    np.testing.assert_array_equal(full, np.concatenate([pre, suf], axis=2))
    np.testing.assert_array_equal(zf, zs)

def _frame_den_matrix(q, k, beta, gf, S, reverse):
    """Frame-rule denominator per (batch, head) as matrix products: z is a
    K-vector; a frame's write is z <- e^{g_f} z, z <- z + K_f^T diag(beta_f)
    (1 - K_f z) with z the post-decay pre-frame state; den = Q_f z. Forward:
    frame f reads frames 0..f. Reverse: frame f reads frames F-1 down to f+1,
    each decayed by its own gate before its write (no self term)."""
    B, T, H, K = q.shape
    F = T // S
    gf = np.asarray(gf, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    out = np.zeros((B, H, T))
    for b in range(B):
        for h in range(H):
            def write(z, f):
                rows = slice(f * S, (f + 1) * S)
                Kf = k[b, rows, h]
                zp = np.exp(gf[b, f, h]) * z
                return zp + Kf.T @ (beta[b, rows, h] * (1.0 - Kf @ zp))
            z = np.zeros(K)
            order = range(F - 1, -1, -1) if reverse else range(F)
            for f in order:
                rows = slice(f * S, (f + 1) * S)
                if not reverse:
                    z = write(z, f)
                out[b, h, rows] = q[b, rows, h] @ z
                if reverse:
                    z = write(z, f)
    return out


@pytest.mark.parametrize("reverse", [False, True])
def test_frame_den_matrix_form(reverse):
    B, F, S, H, K, V = 2, 5, 3, 2, 4, 1
    q, k, _, beta, gf = _frame_rand(41, B, F, S, H, K, V)
    got = oracle.frame_den(q, k, beta, gf, S, reverse=reverse)
    want = _frame_den_matrix(q, k, beta, gf, S, reverse)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    other = _frame_den_matrix(q, k, beta, gf, S, not reverse)
    assert np.abs(got - other).max() > 1e-3


def _rms_relu(x, scale):
    """Full-channel RMSNorm (eps 1e-5, weight 1) over the H*D channels of
    each token, then ReLU, then * scale, written out in numpy."""
    ms = (x * x).mean(axis=(2, 3), keepdims=True)
    return np.maximum(x / np.sqrt(ms + 1e-5), 0.0) * scale


def test_forward_glue_bidirectional_chunk_causal_merge():
    """oracle.forward on a bidirectional workload (chunk-causal backward gates
    and a gate for the merge) equals the pieces put together by hand: the
    prep in numpy, the causal scan plus the reverse scan with the backward
    gates, both denominators, and num / (den + eps) * silu(gate)."""
    import workloads
    w = workloads.make_video(1, 24, 2, 8, seed=3, reset_every=8, merge=True)
    res = oracle.forward(w)
    qn = _rms_relu(w.q.values.astype(np.float64), 1.0)
    kn = _rms_relu(w.k.values.astype(np.float64), 8 ** -0.5)
    v = w.v.values.astype(np.float64)
    of, _ = oracle.scan(qn, kn, v, w.beta, g=w.g)
    orv, _ = oracle.scan(qn, kn, v, w.beta_bwd, g=w.g_bwd, reverse=True)
    num = of + orv
    den = (oracle.den(qn, kn, w.beta, g=w.g)
           + oracle.den(qn, kn, w.beta_bwd, g=w.g_bwd, reverse=True))
    np.testing.assert_allclose(res["out"], num, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(res["den"], den, rtol=1e-12, atol=1e-12)
    x = w.gate.values.astype(np.float64)
    merged = num / (den.transpose(0, 2, 1)[..., None] + w.eps) * (x / (1.0 + np.exp(-x)))
    np.testing.assert_allclose(res["merged"], merged, rtol=1e-12, atol=1e-12)
    # the backward gates matter here: the same sum with the forward gates differs
    orv_plain, _ = oracle.scan(qn, kn, v, w.beta, g=w.g, reverse=True)
    assert np.abs(of + orv_plain - num).max() > 1e-3


def test_forward_glue_frame_bidirectional():
    """oracle.forward on a frame-causal bidirectional workload equals both
    directions of the frame rule and both frame denominators summed, with the
    numpy prep; each direction checked against the matrix forms."""
    import workloads
    w = workloads.make_video(1, 12, 2, 8, seed=4, frame=4)
    res = oracle.forward(w)
    qn = _rms_relu(w.q.values.astype(np.float64), 1.0)
    kn = _rms_relu(w.k.values.astype(np.float64), 8 ** -0.5)
    v = w.v.values.astype(np.float64)
    of, _ = oracle.frame_scan(qn, kn, v, w.beta, w.g_frame, 4)
    orv, _ = oracle.frame_scan(qn, kn, v, w.beta, w.g_frame, 4, reverse=True)
    np.testing.assert_allclose(res["out"], of + orv, rtol=1e-12, atol=1e-12)
    den = (_frame_den_matrix(qn, kn, w.beta, w.g_frame, 4, False)
           + _frame_den_matrix(qn, kn, w.beta, w.g_frame, 4, True))
    np.testing.assert_allclose(res["den"], den, rtol=1e-12, atol=1e-12)
