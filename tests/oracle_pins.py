"""Pins for the fp64 oracle: each checks it against something other than itself.

Sources of truth used here (none of them is the oracle's own formula retyped):
  * numpy.convolve / scipy.special.expit for the conv + SiLU step;
  * one-hot channel probes for the Q/K/V split and the reverse-GQA mapping
    (MNN "Qwen3.5" page, section 1.3: repeat_interleave, not tiling);
  * numpy.linalg.norm for the L2 normalisation and the 1/sqrt(d_k) scale;
  * closed forms of the gated delta rule (section 1.2, Step 5) in its special
    cases: g=0 & beta=0 (constant memory), unit key & beta=1 (exact recall),
    exp(g)=0 (memory reset), basis keys (row overwrite);
  * an exact rational expansion of the recurrence,
        S_t = prod_r M_r S_0 + sum_s prod_{r>s} M_r beta_s k_s v_s^T,
        M_r = alpha_r (I - beta_r k_r k_r^T),
    evaluated with fractions.Fraction on tiny shapes;
  * the contraction bound ||S_t|| <= alpha_t ||S_{t-1}|| + beta_t ||v_t|| for
    unit keys and beta in (0, 1].
Each pin is a plain function that raises AssertionError; tests/test_oracle_pins.py
runs them, and tests/test_oracle_mutations.py runs them against deliberately
broken copies of the oracle to show that each plausible mistake is caught.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import scipy.special

import oracle


def _rng(seed):
    return np.random.default_rng(seed)


def _silu(a):
    return a * scipy.special.expit(a)


def _close(a, b, rtol=1e-13, atol=1e-14, what=""):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    assert np.allclose(a, b, rtol=rtol, atol=atol), f"{what}: max diff {np.max(np.abs(a - b))}"


# ----------------------------------------------------------------------------
# Step 1: causal conv + SiLU
# ----------------------------------------------------------------------------

def pin_conv_numpy_convolve():
    r = _rng(1)
    D, K, L = 5, 4, 9
    x, w, st = r.normal(size=(D, L)), r.normal(size=(D, K)), r.normal(size=(D, K - 1))
    y, st_out, _ = oracle.conv1d_silu(x, w, st)
    for d in range(D):
        xp = np.concatenate([st[d], x[d]])
        pre = np.convolve(xp, w[d][::-1], mode="valid")     # cross-correlation
        _close(y[d], _silu(pre), what="conv vs numpy.convolve")
        _close(st_out[d], xp[-(K - 1):], rtol=0, atol=0, what="conv state tail")


def pin_conv_newest_tap():
    """An impulse at time t0 reaches y[t0] through w[K-1] (the newest tap)."""
    D, K, L, t0 = 2, 4, 8, 2
    x = np.zeros((D, L)); x[:, t0] = 1.0
    w = np.array([[1.0, 2.0, 3.0, 4.0], [-0.5, 0.25, 0.75, -1.5]])
    y, _, _ = oracle.conv1d_silu(x, w, np.zeros((D, K - 1)))
    for d in range(D):
        for j in range(K):
            _close(y[d, t0 + j], _silu(w[d, K - 1 - j]), what="impulse response")
        _close(y[d, :t0], np.zeros(t0), rtol=0, atol=0, what="causality")


def pin_conv_k1_is_silu():
    r = _rng(2)
    x = r.normal(size=(3, 7))
    y, st, _ = oracle.conv1d_silu(x, np.ones((3, 1)), np.zeros((3, 0)))
    _close(y, _silu(x), what="K=1, w=1")
    assert st.shape == (3, 0)


def pin_conv_short_sequence_shift():
    """L < K-1: the window shifts only partly."""
    r = _rng(3)
    D, K = 4, 4
    st = r.normal(size=(D, K - 1))
    for L in (1, 2, 3, 5):
        x = r.normal(size=(D, L))
        _, st_out, snap = oracle.conv1d_silu(x, r.normal(size=(D, K)), st, snapshots=True)
        xp = np.concatenate([st, x], axis=1)
        _close(st_out, xp[:, -(K - 1):], rtol=0, atol=0, what=f"tail L={L}")
        for t in range(L):
            _close(snap[t], xp[:, t + 1:t + K], rtol=0, atol=0, what=f"snapshot t={t}")


# ----------------------------------------------------------------------------
# Steps 2-4: split, reverse GQA, L2 norm, scale
# ----------------------------------------------------------------------------

def pin_split_one_hot():
    cfg = oracle.Cfg(2, 4, 3, 2, use_qk_l2norm=False)
    Hk, Hv, dk, dv = 2, 4, 3, 2
    f = Hv // Hk
    for c in range(cfg.D):
        y = np.zeros((cfg.D, 1)); y[c, 0] = 1.0
        q, k, v = oracle.split_norm_scale(cfg, y)
        eq, ek, ev = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        if c < Hk * dk:
            hk, i = divmod(c, dk)
            eq[0, hk * f:(hk + 1) * f, i] = 1.0 / np.sqrt(dk)
        elif c < 2 * Hk * dk:
            hk, i = divmod(c - Hk * dk, dk)
            ek[0, hk * f:(hk + 1) * f, i] = 1.0
        else:
            h, j = divmod(c - 2 * Hk * dk, dv)
            ev[0, h, j] = 1.0
        _close(q, eq, what=f"q one-hot c={c}")
        _close(k, ek, rtol=0, atol=0, what=f"k one-hot c={c}")
        _close(v, ev, rtol=0, atol=0, what=f"v one-hot c={c}")


def pin_gqa_interleave_not_tile():
    """Value heads 2m and 2m+1 share key head m (repeat_interleave); tiling would pair h and h+Hk."""
    r = _rng(4)
    cfg = oracle.Cfg(2, 4, 4, 3)
    q, k, _ = oracle.split_norm_scale(cfg, r.normal(size=(cfg.D, 3)))
    _close(q[:, 0], q[:, 1], rtol=0, atol=0, what="q heads 0,1 share")
    _close(k[:, 2], k[:, 3], rtol=0, atol=0, what="k heads 2,3 share")
    assert np.max(np.abs(q[:, 0] - q[:, 2])) > 1e-3, "heads 0 and 2 must differ"


def pin_l2norm_numpy():
    r = _rng(5)
    cfg = oracle.Cfg(2, 4, 5, 3, use_qk_l2norm=True, l2norm_eps=1e-6)
    L = 4
    y = r.normal(size=(cfg.D, L))
    q, k, _ = oracle.split_norm_scale(cfg, y)
    for t in range(L):
        for h in range(4):
            hk = h // 2
            yq = y[hk * 5:(hk + 1) * 5, t]
            yk = y[10 + hk * 5:10 + (hk + 1) * 5, t]
            eq = yq / np.sqrt(np.linalg.norm(yq) ** 2 + 1e-6) / np.sqrt(5)
            ek = yk / np.sqrt(np.linalg.norm(yk) ** 2 + 1e-6)
            _close(q[t, h], eq, what="q norm+scale")
            _close(k[t, h], ek, what="k norm")


def pin_l2norm_eps0_unit():
    r = _rng(6)
    cfg = oracle.Cfg(1, 2, 8, 4, use_qk_l2norm=True, l2norm_eps=0.0)
    q, k, _ = oracle.split_norm_scale(cfg, r.normal(size=(cfg.D, 6)))
    _close(np.linalg.norm(q, axis=-1), np.full((6, 2), 1 / np.sqrt(8)), what="|q| = 1/sqrt(dk)")
    _close(np.linalg.norm(k, axis=-1), np.ones((6, 2)), what="|k| = 1")


def pin_no_l2norm_scale_only():
    r = _rng(7)
    cfg = oracle.Cfg(1, 1, 4, 2, use_qk_l2norm=False)
    y = r.normal(size=(cfg.D, 3))
    q, k, v = oracle.split_norm_scale(cfg, y)
    _close(q[:, 0], y[0:4].T / 2.0, what="q scale only")
    _close(k[:, 0], y[4:8].T, rtol=0, atol=0, what="k untouched")
    _close(v[:, 0], y[8:10].T, rtol=0, atol=0, what="v untouched")


# ----------------------------------------------------------------------------
# Step 5: gated delta rule
# ----------------------------------------------------------------------------

def _qkv(r, L=5, H=2, dk=3, dv=4, unit_k=False):
    q = r.normal(size=(L, H, dk)); k = r.normal(size=(L, H, dk)); v = r.normal(size=(L, H, dv))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    S0 = r.normal(size=(H, dk, dv))
    return q, k, v, S0


def pin_rule_frozen_memory():
    """g=0, beta=0: S stays S_0 and o_t = S_0^T q_t."""
    r = _rng(10)
    q, k, v, S0 = _qkv(r)
    L, H = q.shape[:2]
    o, S, _ = oracle.delta_rule(q, k, v, np.zeros((L, H)), np.zeros((L, H)), S0)
    _close(S, S0, rtol=0, atol=0, what="S constant")
    _close(o, np.einsum("hij,thi->thj", S0, q), what="o = S0^T q")


def pin_rule_exact_recall():
    """Unit key, beta=1: after the update S^T k_t = v_t exactly."""
    r = _rng(11)
    q, k, v, S0 = _qkv(r, unit_k=True)
    L, H = q.shape[:2]
    g = -r.uniform(0, 2, size=(L, H))
    _, _, snap = oracle.delta_rule(q, k, v, g, np.ones((L, H)), S0, snapshots=True)
    for t in range(L):
        _close(np.einsum("hij,hi->hj", snap[t], k[t]), v[t], rtol=1e-12, atol=1e-12, what=f"recall t={t}")


def pin_rule_reset():
    """exp(g)=0 (g=-inf, or a large negative g underflowing): S_t = beta k v^T, o_t = beta (k.q) v."""
    r = _rng(12)
    q, k, v, S0 = _qkv(r)
    L, H = q.shape[:2]
    beta = r.uniform(0.1, 1.0, size=(L, H))
    for gval in (-np.inf, -1000.0):
        o, _, snap = oracle.delta_rule(q, k, v, np.full((L, H), gval), beta, S0, snapshots=True)
        for t in range(L):
            _close(snap[t], beta[t][:, None, None] * np.einsum("hi,hj->hij", k[t], v[t]), what="reset state")
            _close(o[t], (beta[t] * np.einsum("hi,hi->h", k[t], q[t]))[:, None] * v[t], what="reset output")


def pin_rule_basis_key_overwrite():
    """g=0, beta=1, k=e_i: row i of S becomes v_t; other rows are untouched."""
    r = _rng(13)
    L, H, dk, dv = 6, 2, 3, 4
    q, _, v, S0 = _qkv(r, L, H, dk, dv)
    rows = r.integers(0, dk, size=(L, H))
    k = np.zeros((L, H, dk))
    for t in range(L):
        for h in range(H):
            k[t, h, rows[t, h]] = 1.0
    _, _, snap = oracle.delta_rule(q, k, v, np.zeros((L, H)), np.ones((L, H)), S0, snapshots=True)
    prev = S0.copy()
    for t in range(L):
        exp_ = prev.copy()
        for h in range(H):
            exp_[h, rows[t, h]] = v[t, h]
        _close(snap[t], exp_, rtol=0, atol=1e-15, what=f"overwrite t={t}")
        prev = exp_


def _frac_vec(r, n, den=7):
    return [Fraction(int(x), den) for x in r.integers(-den, den + 1, size=n)]


def pin_rule_exact_rational_expansion():
    """Tiny shapes (d_k=2, d_v=3, L=4, two heads) checked against the exact rational
    expansion of the recurrence; the oracle gets g = log(alpha)."""
    r = _rng(14)
    H, dk, dv, L = 2, 2, 3, 4
    qF = [[_frac_vec(r, dk) for _ in range(H)] for _ in range(L)]
    kF = [[_frac_vec(r, dk) for _ in range(H)] for _ in range(L)]
    vF = [[_frac_vec(r, dv) for _ in range(H)] for _ in range(L)]
    aF = [[Fraction(int(r.integers(1, 9)), 8) for _ in range(H)] for _ in range(L)]
    bF = [[Fraction(int(r.integers(1, 6)), 5) for _ in range(H)] for _ in range(L)]
    S0F = [[[Fraction(int(x), 3) for x in r.integers(-3, 4, size=dv)] for _ in range(dk)] for _ in range(H)]

    def mm(A, B):
        return [[sum(A[i][m] * B[m][j] for m in range(len(B))) for j in range(len(B[0]))] for i in range(len(A))]

    def eye(n):
        return [[Fraction(int(i == j)) for j in range(n)] for i in range(n)]

    def M(t, h):   # alpha (I - beta k k^T)
        k = kF[t][h]
        return [[aF[t][h] * ((1 if i == j else 0) - bF[t][h] * k[i] * k[j]) for j in range(dk)] for i in range(dk)]

    f64 = lambda X: np.array([[float(x) for x in row] for row in X])
    q = np.array([[[float(x) for x in qF[t][h]] for h in range(H)] for t in range(L)])
    k = np.array([[[float(x) for x in kF[t][h]] for h in range(H)] for t in range(L)])
    v = np.array([[[float(x) for x in vF[t][h]] for h in range(H)] for t in range(L)])
    g = np.log(np.array([[float(aF[t][h]) for h in range(H)] for t in range(L)]))
    beta = np.array([[float(bF[t][h]) for h in range(H)] for t in range(L)])
    S0 = np.array([f64(S0F[h]) for h in range(H)])
    o, S, snap = oracle.delta_rule(q, k, v, g, beta, S0, snapshots=True)
    for h in range(H):
        for t in range(L):
            P = eye(dk)
            for rr in range(t + 1):
                P = mm(M(rr, h), P)                   # M_t ... M_0
            St = mm(P, S0F[h])
            for s in range(t + 1):
                Q = eye(dk)
                for rr in range(s + 1, t + 1):
                    Q = mm(M(rr, h), Q)
                kv = [[bF[s][h] * kF[s][h][i] * vF[s][h][j] for j in range(dv)] for i in range(dk)]
                add = mm(Q, kv)
                St = [[St[i][j] + add[i][j] for j in range(dv)] for i in range(dk)]
            ot = [sum(St[i][j] * qF[t][h][i] for i in range(dk)) for j in range(dv)]
            _close(snap[t, h], f64(St), rtol=1e-12, atol=1e-12, what=f"exact S t={t} h={h}")
            _close(o[t, h], [float(x) for x in ot], rtol=1e-12, atol=1e-12, what=f"exact o t={t} h={h}")
        _close(S[h], snap[L - 1, h], rtol=0, atol=0, what="final = last snapshot")


def pin_rule_contraction():
    r = _rng(15)
    q, k, v, S0 = _qkv(r, L=12, H=3, dk=6, dv=5, unit_k=True)
    L, H = q.shape[:2]
    g = -r.uniform(0, 1.5, size=(L, H))
    beta = r.uniform(0.01, 1.0, size=(L, H))
    _, _, snap = oracle.delta_rule(q, k, v, g, beta, S0, snapshots=True)
    prev = S0
    for t in range(L):
        for h in range(H):
            lhs = np.linalg.norm(snap[t, h], 2)
            rhs = np.exp(g[t, h]) * np.linalg.norm(prev[h], 2) + beta[t, h] * np.linalg.norm(v[t, h])
            assert lhs <= rhs * (1 + 1e-12), f"contraction t={t} h={h}: {lhs} > {rhs}"
        prev = snap[t]


# ----------------------------------------------------------------------------
# All five steps
# ----------------------------------------------------------------------------

def _seq(r, cfg, L):
    D, K, H = cfg.D, cfg.conv_kernel, cfg.num_v_heads
    return dict(x=r.normal(size=(D, L)), w=r.normal(scale=0.5, size=(D, K)),
                conv_in=r.normal(size=(D, K - 1)),
                S_in=r.normal(scale=0.02, size=(H, cfg.head_k_dim, cfg.head_v_dim)),
                g=-np.logaddexp(0, r.normal(size=(L, H))), beta=scipy.special.expit(r.normal(size=(L, H))))


def pin_forward_is_composition():
    r = _rng(20)
    cfg = oracle.Cfg(2, 4, 4, 3)
    s = _seq(r, cfg, 6)
    out = oracle.forward_sequence(cfg, s["x"], s["w"], s["conv_in"], s["S_in"], s["g"], s["beta"])
    y, conv, _ = oracle.conv1d_silu(s["x"], s["w"], s["conv_in"])
    q, k, v = oracle.split_norm_scale(cfg, y)
    o, S, _ = oracle.delta_rule(q, k, v, s["g"], s["beta"], s["S_in"])
    _close(out["o"], o, rtol=0, atol=0, what="o")
    _close(out["S"], S, rtol=0, atol=0, what="S")
    _close(out["conv"], conv, rtol=0, atol=0, what="conv")


def pin_forward_split_equals_whole():
    """Two calls with carried conv and SSM state equal one call (section 1.4: the
    states persist across steps)."""
    r = _rng(21)
    cfg = oracle.Cfg(2, 4, 4, 3)
    s = _seq(r, cfg, 11)
    whole = oracle.forward_sequence(cfg, s["x"], s["w"], s["conv_in"], s["S_in"], s["g"], s["beta"])
    for cut in (1, 2, 5, 10):
        a = oracle.forward_sequence(cfg, s["x"][:, :cut], s["w"], s["conv_in"], s["S_in"], s["g"][:cut], s["beta"][:cut])
        b = oracle.forward_sequence(cfg, s["x"][:, cut:], s["w"], a["conv"], a["S"], s["g"][cut:], s["beta"][cut:])
        _close(np.concatenate([a["o"], b["o"]]), whole["o"], rtol=0, atol=0, what=f"o cut={cut}")
        _close(b["S"], whole["S"], rtol=0, atol=0, what=f"S cut={cut}")
        _close(b["conv"], whole["conv"], rtol=0, atol=0, what=f"conv cut={cut}")


def pin_forward_snapshots_are_prefix_runs():
    r = _rng(22)
    cfg = oracle.Cfg(1, 2, 4, 4)
    s = _seq(r, cfg, 4)
    full = oracle.forward_sequence(cfg, s["x"], s["w"], s["conv_in"], s["S_in"], s["g"], s["beta"], snapshots=True)
    for t in range(4):
        p = oracle.forward_sequence(cfg, s["x"][:, :t + 1], s["w"], s["conv_in"], s["S_in"], s["g"][:t + 1], s["beta"][:t + 1])
        _close(full["S_snap"][t], p["S"], rtol=0, atol=0, what=f"S snap {t}")
        _close(full["conv_snap"][t], p["conv"], rtol=0, atol=0, what=f"conv snap {t}")


# ---- gate parameterisation (section 1.2) -------------------------------------

def pin_gate_beta_closed_forms():
    # softplus(0) = ln 2, sigmoid(0) = 1/2, sigmoid(ln 3) = 3/4, exp(ln 2) = 2
    a = np.array([[0.0, -0.5, 2.0]])
    b = np.array([[0.0, np.log(3.0), -np.log(3.0)]])
    A_log = np.array([0.0, np.log(2.0), 0.0])
    dt_bias = np.array([0.0, 0.5, -2.0])
    g, beta = oracle.gate_beta(a, b, A_log, dt_bias)
    _close(g, [[-np.log(2.0), -2.0 * np.log(2.0), -np.log(2.0)]], what="gate closed forms")
    _close(beta, [[0.5, 0.75, 0.25]], what="beta closed forms")


def pin_gate_beta_library():
    r = _rng(41)
    a, b = r.normal(0, 3, (6, 5)), r.normal(0, 3, (6, 5))
    A_log, dt_bias = r.normal(0, 1, 5), r.normal(0, 1, 5)
    g, beta = oracle.gate_beta(a, b, A_log, dt_bias)
    _close(g, -np.exp(A_log) * np.logaddexp(0.0, a + dt_bias), what="gate vs numpy.logaddexp")
    _close(beta, scipy.special.expit(b), what="beta vs scipy expit")
    assert np.all(g <= 0.0) and np.all(np.exp(g) <= 1.0), "decay above 1"


def pin_gate_large_argument():
    # softplus(x) -> x for large x, -> e^x for very negative x
    g, _ = oracle.gate_beta(np.array([[60.0, -40.0]]), np.zeros((1, 2)), np.array([0.5, 0.0]), np.array([0.0, 0.0]))
    _close(g[0, 0], -np.exp(0.5) * 60.0, what="softplus large x")
    _close(g[0, 1], -np.exp(-40.0), rtol=1e-12, atol=0.0, what="softplus very negative x")


# ---- gated RMSNorm (section 2) ------------------------------------------------

def pin_gated_rmsnorm_numpy():
    r = _rng(43)
    o, z = r.normal(0, 2, (5, 3, 8)), r.normal(0, 2, (5, 3, 8))
    w = r.normal(1, 0.3, 8)
    y = oracle.gated_rmsnorm(o, z, w, 1e-6)
    rms = np.linalg.norm(o, axis=-1, keepdims=True) / np.sqrt(8.0)
    ref = w * (o / np.sqrt(rms ** 2 + 1e-6)) * _silu(z)
    _close(y, ref, what="gated RMSNorm vs numpy")


def pin_gated_rmsnorm_closed_forms():
    # a constant row c with unit weight and eps = 0 normalises to sign(c); z = 0 gates to 0;
    # silu(ln 3) = (3/4) ln 3
    o = np.array([[-2.5] * 4, [3.0, -3.0, 3.0, -3.0]])
    z = np.array([[np.log(3.0)] * 4, [0.0, 1.0, 0.0, 1.0]])
    y = oracle.gated_rmsnorm(o, z, np.ones(4), 0.0)
    _close(y[0], [-0.75 * np.log(3.0)] * 4, what="constant row")
    _close(y[1], [0.0, -scipy.special.expit(1.0), 0.0, -scipy.special.expit(1.0)], what="z = 0 and z = 1")
    # eps: a row of zeros stays finite and zero
    y0 = oracle.gated_rmsnorm(np.zeros((1, 4)), np.ones((1, 4)), np.ones(4), 1e-6)
    _close(y0, np.zeros((1, 4)), what="zero row")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
