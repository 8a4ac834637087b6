"""The rearranged recurrences of the decode/verify and resident-prefill kernels, emulated
in fp64 on the CPU and held against the oracle's literal order (MNN "Qwen3.5" page,
section 1.2, step 5: decay, predict, error, update, read-out as separate passes):

- the single pass of the streaming kernels, which reads and writes each state element
  once per token: a = (alpha S)^T k, delta = beta (v - a), o = alpha S^T q + delta (k.q),
  S' = alpha S + k delta^T;
- the 8-token blocks of the resident prefill, where every token's products with the
  block's starting state S0 are independent:
  a_t = gamma_t (S0^T k_t) + sum_{s<t} e^{G_t - G_s} (k_s.k_t) delta_s,
  o_t = gamma_t (S0^T q_t) + sum_{s<=t} e^{G_t - G_s} (k_s.q_t) delta_s,
  S_end = gamma_last S0 + sum_s e^{G_last - G_s} k_s delta_s^T.
Both must equal the literal recurrence to rounding.
"""
import numpy as np
import pytest

import oracle


def _inputs(seed, L=40, dk=8, dv=6):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((L, dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    q = rng.standard_normal((L, dk)) / np.sqrt(dk)
    v = rng.standard_normal((L, dv))
    g = -np.log1p(np.exp(rng.standard_normal(L)))  # -softplus(N(0,1))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(L)))
    S0 = 0.3 * rng.standard_normal((dk, dv))
    return q, k, v, g, beta, S0


def _oracle(q, k, v, g, beta, S0):
    o, S, _ = oracle.delta_rule(q[:, None], k[:, None], v[:, None], g[:, None], beta[:, None], S0[None])
    return o[:, 0], S[0]


def _single_pass(q, k, v, g, beta, S0):
    S = S0.copy()
    o = np.zeros((len(q), v.shape[1]))
    for t in range(len(q)):
        al = np.exp(g[t])
        a = al * (S.T @ k[t])
        d = beta[t] * (v[t] - a)
        o[t] = al * (S.T @ q[t]) + d * (k[t] @ q[t])
        S = al * S + np.outer(k[t], d)
    return o, S


def _blocks(q, k, v, g, beta, S0, B=8):
    S = S0.copy()
    o = np.zeros((len(q), v.shape[1]))
    for b0 in range(0, len(q), B):
        idx = range(b0, min(len(q), b0 + B))
        G = np.cumsum(g[b0:b0 + B])
        Sk, Sq = [S.T @ k[t] for t in idx], [S.T @ q[t] for t in idx]
        d = []
        for i, t in enumerate(idx):
            a = np.exp(G[i]) * Sk[i] + sum(np.exp(G[i] - G[j]) * (k[s] @ k[t]) * d[j] for j, s in enumerate(idx) if j < i)
            d.append(beta[t] * (v[t] - a))
            o[t] = np.exp(G[i]) * Sq[i] + sum(np.exp(G[i] - G[j]) * (k[s] @ q[t]) * d[j]
                                                for j, s in enumerate(idx) if j <= i)
        S = np.exp(G[-1]) * S + sum(np.exp(G[-1] - G[j]) * np.outer(k[s], d[j]) for j, s in enumerate(idx))
    return o, S


@pytest.mark.parametrize("form", [_single_pass, _blocks], ids=["single_pass", "blocks_of_8"])
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_rearranged_recurrence_equals_literal_order(oracle_mod, form, seed):
    q, k, v, g, beta, S0 = _inputs(seed, L=37)  # a ragged last block
    o_ref, S_ref = _oracle(q, k, v, g, beta, S0)
    o, S = form(q, k, v, g, beta, S0)
    scale = np.sqrt(np.mean(o_ref ** 2))
    assert np.max(np.abs(o - o_ref)) <= 1e-12 * scale
    assert np.linalg.norm(S - S_ref) <= 1e-12 * np.linalg.norm(S_ref)


def test_forms_see_a_dropped_term(oracle_mod):
    """The comparison is sharp enough to catch a plausible slip: dropping the (k.q) term
    of the single pass (reading the output before the update) moves o far off."""
    q, k, v, g, beta, S0 = _inputs(4, L=12)
    o_ref, _ = _oracle(q, k, v, g, beta, S0)
    S = S0.copy()
    o = np.zeros_like(o_ref)
    for t in range(len(q)):
        al = np.exp(g[t])
        d = beta[t] * (v[t] - al * (S.T @ k[t]))
        o[t] = al * (S.T @ q[t])
        S = al * S + np.outer(k[t], d)
    assert np.max(np.abs(o - o_ref)) > 1e-3 * np.sqrt(np.mean(o_ref ** 2))
