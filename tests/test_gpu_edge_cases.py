"""The recurrence's closed-form cases fed to every CUDA path: decode (both decode
kernels), verify, and both prefill forms.

The gated delta rule (MNN "Qwen3.5" page, section 1.2, Step 5: decay, predict,
error, update, read-out) has four inputs for which the result is known without
running it:

  hold    g = 0, beta = 0: the state never changes and o_t = S0^T q_t;
  recall  unit-norm keys (eps = 0) and beta = 1: after token t, S^T k_t = v_t
          (the update writes v_t exactly into the direction k_t);
  reset   g = -1e4, so exp(g) underflows to 0: after token t, S = beta_t k_t v_t^T
          and o_t = beta_t (k_t . q_t) v_t;
  fade    beta = 0 with a random decay: after token t, S = exp(G_t) S0 with G_t the
          running sum of the log-decays, and o_t = exp(G_t) S0^T q_t.

Each test compares the GPU's outputs and states with the fp64 oracle element by
element at the layer's bar (max|do| <= 2e-3 RMS(o), state relative L2 <= 1e-4),
then checks the case's own property on the GPU's states, with q, k, v taken from
the oracle's steps 1-4 on the same input bits.  Every output and snapshot buffer
carries guard bands that must come back untouched.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_causal_gb300 import binding as gb
from gated_deltanet_linear_causal_gb300 import synth
from gdn_testutil import Guarded, assert_parity, bits, configs, device, f64, state_err, to_dev

pytestmark = pytest.mark.gpu

CASES = ["hold", "recall", "reset", "fade"]
STREAM = synth.Shape(2, 4, 128, 128, 4)   # the persistent bulk-copy decode kernel's shape
SLICE = synth.Shape(2, 4, 64, 64, 4)      # the cluster slice kernel's shape
NARROW = synth.Shape(2, 4, 128, 64, 4)    # chunked prefill with d_v < d_k


def _gates(case, gate, beta):
    """gate/beta arrays (any shape) for a case, from the seeded random ones."""
    gate, beta = np.array(gate, np.float32), np.array(beta, np.float32)
    if case == "hold":
        return np.zeros_like(gate), np.zeros_like(beta)
    if case == "recall":
        return gate, np.ones_like(beta)
    if case == "reset":
        return np.full_like(gate, -1e4), beta
    return (0.2 * gate).astype(np.float32), np.zeros_like(beta)   # fade: slow decay, no writes


def _eps(case):
    return 0.0 if case == "recall" else 1e-6


def _qkv_tokens(ocfg, x, w, conv_in):
    """Steps 1-4 of the oracle on one sequence x [D, L]: q, k [L, H, dk], v [L, H, dv]."""
    y, _, _ = oracle.conv1d_silu(x, w, conv_in)
    return oracle.split_norm_scale(ocfg, y)


def _check_property(case, states, S0, q, k, v, g, beta, what):
    """states[t]: the GPU state after token t (or None to skip); S0 the state before
    token 0; q, k, v, g, beta of the tokens (fp64, [L, H, ..])."""
    G = np.cumsum(np.asarray(g, np.float64), axis=0)
    for t, S in enumerate(states):
        if S is None:
            continue
        if case == "hold":
            assert np.array_equal(bits(S), bits(torch.from_numpy(np.ascontiguousarray(S0, np.float32)))), \
                f"{what}: state changed at token {t}"
            continue
        Sd = f64(S)
        if case == "recall":
            got = np.einsum("hij,hi->hj", Sd, k[t])
            err = np.max(np.abs(got - v[t])) / np.sqrt(np.mean(v[t] ** 2))
            assert err <= 1e-3, f"{what}: S^T k - v = {err:.3g} RMS(v) at token {t}"
        elif case == "reset":
            ref = beta[t][:, None, None] * np.einsum("hi,hj->hij", k[t], v[t])
            assert state_err(Sd, ref) <= 1e-4, f"{what}: S != beta k v^T at token {t}"
        else:
            ref = np.exp(G[t])[:, None, None] * S0
            assert state_err(Sd, ref) <= 1e-4, f"{what}: S != exp(G) S0 at token {t}"


# ---------------------------------------------------------------------------
# decode and verify
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [STREAM, SLICE], ids=["stream", "slice"])
@pytest.mark.parametrize("case", CASES)
def test_decode_closed_forms(case, shape):
    dev = device()
    cfg, ocfg = configs(shape, "bf16", eps=_eps(case))
    B, steps = 3, 3
    st = synth.decode_state(61, B, shape)
    w_d, conv_d, S_d = to_dev(st["conv_weight"], dev), to_dev(st["conv_state"], dev), to_dev(st["ssm_state"], dev)
    w64 = f64(st["conv_weight"])
    conv_r, S_r = f64(st["conv_state"]), st["ssm_state"].astype(np.float64)
    out = Guarded((B, shape.num_v_heads, shape.head_v_dim), torch.float32, dev)
    for step in range(steps):
        d = synth.decode_step(61, step, B, shape)
        gate, beta = _gates(case, d["gate"], d["beta"])
        S_before = f64(S_d)
        gb.gdn_forward_decode(cfg, B, to_dev(d["qkv"], dev), w_d, to_dev(gate, dev), to_dev(beta, dev), conv_d, S_d,
                              out.t)
        o_r, conv_next, S_r = oracle.decode(ocfg, f64(d["qkv"]), w64, gate, beta, conv_r, S_r)
        torch.cuda.synchronize()
        assert_parity(f64(out.t), o_r, f64(S_d), S_r, what=f"{case} step {step}")
        for b in range(B):
            q, k, v = _qkv_tokens(ocfg, f64(d["qkv"][b])[:, None], w64, conv_r[b])
            _check_property(case, [S_d[b]], S_before[b], q, k, v, gate[b][None], beta[b][None],
                            f"{case} step {step} seq {b}")
        conv_r = conv_next
        out.check(f"{case} step {step}")
    assert np.array_equal(f64(conv_d), conv_r)


@pytest.mark.parametrize("shape", [STREAM, SLICE], ids=["stream", "slice"])
@pytest.mark.parametrize("case", CASES)
def test_verify_closed_forms(case, shape):
    dev = device()
    cfg, ocfg = configs(shape, "bf16", eps=_eps(case))
    B, L = 3, 4
    v = synth.verify_block(62, B, L, shape)
    gate, beta = _gates(case, v["gate"], v["beta"])
    H, dk, dv, D = shape.num_v_heads, shape.head_k_dim, shape.head_v_dim, shape.D
    csnap = Guarded((B, L, D, shape.conv_kernel - 1), torch.bfloat16, dev)
    ssnap = Guarded((B, L, H, dk, dv), torch.float32, dev)
    out = Guarded((B, L, H, dv), torch.float32, dev)
    gb.gdn_forward_verify(cfg, B, L, to_dev(v["qkv"], dev), to_dev(v["conv_weight"], dev), to_dev(gate, dev),
                          to_dev(beta, dev), to_dev(v["conv_state"], dev), to_dev(v["ssm_state"], dev), csnap.t,
                          ssnap.t, out.t)
    w64 = f64(v["conv_weight"])
    o_r, cs_r, ss_r = oracle.verify(ocfg, f64(v["qkv"]), w64, gate, beta, f64(v["conv_state"]), v["ssm_state"])
    torch.cuda.synchronize()
    for t in range(L):
        assert_parity(f64(out.t[:, t]), o_r[:, t], f64(ssnap.t[:, t]), ss_r[:, t], what=f"{case} token {t}")
    assert np.array_equal(f64(csnap.t), cs_r)
    for b in range(B):
        q, k, vv = _qkv_tokens(ocfg, f64(v["qkv"][b]), w64, f64(v["conv_state"][b]))
        _check_property(case, [ssnap.t[b, t] for t in range(L)], v["ssm_state"][b].astype(np.float64), q, k, vv,
                        gate[b], beta[b], f"{case} seq {b}")
    for g_, name in ((csnap, "conv snapshots"), (ssnap, "state snapshots"), (out, "output")):
        g_.check(f"{case} {name}")


# ---------------------------------------------------------------------------
# prefill, both forms
# ---------------------------------------------------------------------------

PREFILL = [(gb.GDN_PREFILL_RESIDENT, SLICE), (gb.GDN_PREFILL_RESIDENT, STREAM),
           (gb.GDN_PREFILL_CHUNKED, STREAM), (gb.GDN_PREFILL_CHUNKED, NARROW)]


@pytest.mark.parametrize("variant,shape", PREFILL,
                         ids=["resident-64", "resident-128", "chunked-128", "chunked-128x64"])
@pytest.mark.parametrize("case", CASES)
def test_prefill_closed_forms(case, variant, shape):
    """Three sequences of 150 (two full 64-token chunks and a ragged tail), 64 and 1 tokens,
    each from its own random state."""
    dev = device()
    cfg, ocfg = configs(shape, "bf16", eps=_eps(case))
    x = synth.varlen_prefill(seed=63, shape=shape, lengths=[150, 64, 1])
    gate, beta = _gates(case, x["gate"], x["beta"])
    x = dict(x, gate=gate, beta=beta)
    cu = x["cu_seqlens"]
    N, T = len(cu) - 1, int(cu[-1])
    conv, S = to_dev(x["conv_state"], dev), to_dev(x["ssm_state"], dev)
    out = Guarded((T, shape.num_v_heads, shape.head_v_dim), torch.float32, dev)
    ws = torch.empty(max(1, gb.gdn_prefill_workspace_size(cfg, N, T, variant)), dtype=torch.uint8, device=dev)
    gb.gdn_forward_prefill(cfg, N, to_dev(cu, dev), cu, to_dev(x["qkv"], dev), to_dev(x["conv_weight"], dev),
                           to_dev(gate, dev), to_dev(beta, dev), conv, S, out.t, variant, ws)
    w64 = f64(x["conv_weight"])
    o_r, c_r, S_r = oracle.prefill(ocfg, cu, f64(x["qkv"]), w64, gate, beta, f64(x["conv_state"]), x["ssm_state"])
    torch.cuda.synchronize()
    assert_parity(f64(out.t), o_r, f64(S), S_r, what=case)
    assert np.array_equal(f64(conv), c_r)
    out.check(case)
    for n in range(N):
        a, b = int(cu[n]), int(cu[n + 1])
        q, k, v = _qkv_tokens(ocfg, f64(x["qkv"][:, a:b]), w64, f64(x["conv_state"][n]))
        states = [None] * (b - a - 1) + [S[n]]   # the call leaves the state after the last token
        _check_property(case, states, x["ssm_state"][n].astype(np.float64), q, k, v, gate[a:b], beta[a:b],
                        f"{case} seq {n}")
