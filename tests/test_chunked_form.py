"""The chunked (WY) form of the gated delta rule that the tensor-core prefill computes,
emulated with numpy on the CPU and held against the oracle's literal recurrence (MNN
"Qwen3.5" page, section 1.2, step 5):

- with fp64 products it is the same recurrence, to rounding: this pins the algebra the
  kernels use (T = (I + A)^-1, W, u, U = u - W S0, O = Q~ S0 + P U, S_end = g S0 + K~^T U);
- with every product taken as a three-term bf16 hi/lo split it meets the layer's
  tolerances (max|do| <= 2e-3 RMS(o), state relative L2 <= 1e-4);
- with single-pass bf16 operands it does not, which is why the kernels carry the split.
"""
import numpy as np
import pytest

import oracle
from gated_deltanet_linear_causal_gb300 import synth
from gdn_testutil import f64

O_TOL, S_TOL = 2e-3, 1e-4


def _bf16(x):
    return synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(np.asarray(x, np.float32))).astype(np.float64)


def _prod(a, b, mode):
    if mode == "f64":
        return a @ b
    if mode == "bf16":
        return _bf16(a) @ _bf16(b)
    ah, bh = _bf16(a), _bf16(b)  # "split": x = hi + lo, the lo*lo term dropped
    al, bl = _bf16(a - ah), _bf16(b - bh)
    return ah @ bh + ah @ bl + al @ bh


def _chunked(q, k, v, g, beta, S0, mode, C=64):
    """One head: q, k [L, d_k], v [L, d_v], g, beta [L], S0 [d_k, d_v]."""
    L = q.shape[0]
    S = S0.copy()
    O = np.zeros((L, v.shape[1]))
    for c0 in range(0, L, C):
        sl = slice(c0, min(L, c0 + C))
        n = sl.stop - sl.start
        Q, K, V, b = q[sl], k[sl], v[sl], beta[sl]
        G = np.cumsum(g[sl])
        gam = np.exp(G)
        dec = np.exp(G[:, None] - G[None, :])
        strict, lower = np.tril(np.ones((n, n)), -1), np.tril(np.ones((n, n)))
        A = b[:, None] * dec * _prod(K, K.T, mode) * strict
        T = np.linalg.inv(np.eye(n) + A)
        W = _prod(T, (b * gam)[:, None] * K, mode)
        u = _prod(T, b[:, None] * V, mode)
        U = u - _prod(W, S, mode)
        P = _prod(Q, K.T, mode) * dec * lower
        O[sl] = _prod(gam[:, None] * Q, S, mode) + _prod(P, U, mode)
        Kt = np.exp(G[-1] - G)[:, None] * K
        S = gam[-1] * S + _prod(Kt.T, U, mode)
    return O, S


@pytest.fixture(scope="module")
def head(oracle_mod):
    """Value head 5 of the long-prefill workload (slow decay, zero state), first 1024 tokens."""
    shape = synth.PRODUCTION
    x = synth.long_prefill(seed=3, L=1024)
    Hk, dk, dv, f, h = shape.num_k_heads, shape.head_k_dim, shape.head_v_dim, shape.num_v_heads // shape.num_k_heads, 5
    hk = h // f
    ch = np.r_[hk * dk:(hk + 1) * dk, Hk * dk + hk * dk:Hk * dk + (hk + 1) * dk,
               2 * Hk * dk + h * dv:2 * Hk * dk + (h + 1) * dv]
    K = shape.conv_kernel
    y = oracle.conv1d_silu(f64(x["qkv"][ch]), f64(x["conv_weight"][ch]), np.zeros((len(ch), K - 1)))[0]
    q, k, v = oracle.split_norm_scale(oracle.Cfg(1, 1, dk, dv, K), y)
    g, b = x["gate"][:, h].astype(np.float64), x["beta"][:, h].astype(np.float64)
    S0 = np.zeros((dk, dv))
    o_ref, S_ref = oracle.delta_rule(q, k, v, g[:, None], b[:, None], S0[None])[:2]
    return dict(q=q[:, 0], k=k[:, 0], v=v[:, 0], g=g, b=b, S0=S0, o=o_ref[:, 0], S=S_ref[0])


def _errors(hd, mode):
    O, S = _chunked(hd["q"], hd["k"], hd["v"], hd["g"], hd["b"], hd["S0"], mode)
    eo = np.max(np.abs(O - hd["o"])) / np.sqrt(np.mean(hd["o"] ** 2))
    es = np.linalg.norm(S - hd["S"]) / np.linalg.norm(hd["S"])
    return eo, es


def test_chunked_form_is_the_recurrence(head):
    eo, es = _errors(head, "f64")
    assert eo < 1e-9 and es < 1e-9, (eo, es)


def test_split_products_meet_the_tolerances(head):
    eo, es = _errors(head, "split")
    assert eo <= O_TOL and es <= S_TOL, (eo, es)


def test_single_pass_bf16_misses_the_output_tolerance(head):
    eo, _ = _errors(head, "bf16")
    assert eo > O_TOL, eo
