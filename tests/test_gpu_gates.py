"""The gate parameterisation of section 1.2 done in the kernels: with A_log and
dt_bias in the config, the gate and beta inputs are the raw projections a and b,
and every path forms gate = -exp(A_log) * softplus(a + dt_bias), beta = sigmoid(b)
itself.  Checked against the fp64 oracle applying the same parameterisation
(oracle.gate_beta) before the layer."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_causal_gb300 import binding as gb
from gated_deltanet_linear_causal_gb300 import synth
from gdn_testutil import assert_parity, bits, device, f64, to_dev

pytestmark = pytest.mark.gpu


def _cfgs(shape, io, raw, dev):
    A, dt = to_dev(raw["A_log"], dev), to_dev(raw["dt_bias"], dev)
    cfg = gb.make_config(shape.num_k_heads, shape.num_v_heads, shape.head_k_dim, shape.head_v_dim,
                         shape.conv_kernel, True, 1e-6, io, A_log=A, dt_bias=dt)
    ocfg = oracle.Cfg(shape.num_k_heads, shape.num_v_heads, shape.head_k_dim, shape.head_v_dim, shape.conv_kernel,
                      True, 1e-6)
    return cfg, ocfg


@pytest.mark.parametrize("shape,io", [(synth.PRODUCTION, "bf16"), (synth.Shape(2, 4, 32, 32, 4), "f32")],
                         ids=["production-stream-kernel", "small-slice-kernel"])
def test_decode_raw_gates(shape, io):
    dev = device()
    batch, steps = (8, 3) if shape is synth.PRODUCTION else (3, 4)
    st = synth.decode_state(61, batch, shape)
    cvt = (lambda a: a) if io == "bf16" else synth.bf16_bits_to_f32
    raw = synth.raw_gates(62, (steps, batch), shape.num_v_heads)
    cfg, ocfg = _cfgs(shape, io, raw, dev)
    g_r, b_r = oracle.gate_beta(raw["a"], raw["b"], raw["A_log"], raw["dt_bias"])
    w = cvt(st["conv_weight"])
    conv_d, S_d = to_dev(cvt(st["conv_state"]), dev), to_dev(st["ssm_state"], dev)
    conv_r, S_r = f64(cvt(st["conv_state"])), st["ssm_state"].astype(np.float64)
    out = torch.empty(batch, shape.num_v_heads, shape.head_v_dim, device=dev)
    for s in range(steps):
        qkv = cvt(synth.decode_step(61, s, batch, shape)["qkv"])
        gb.gdn_forward_decode(cfg, batch, to_dev(qkv, dev), to_dev(w, dev), to_dev(raw["a"][s], dev),
                              to_dev(raw["b"][s], dev), conv_d, S_d, out)
        o_r, conv_r, S_r = oracle.decode(ocfg, f64(qkv), f64(w), g_r[s], b_r[s], conv_r, S_r)
        torch.cuda.synchronize()
        assert_parity(f64(out), o_r, what=f"step {s}")
    assert_parity(f64(out), o_r, f64(S_d), S_r, what="final")


def test_verify_raw_gates_snapshots_equal_decode():
    """Verify with raw gates: snapshot t bitwise equals t+1 decode calls with the same raw
    gates, and the outputs match the oracle."""
    dev = device()
    shape, B, L = synth.PRODUCTION, 4, 3
    v = synth.verify_block(63, B, L, shape)
    raw = synth.raw_gates(64, (B, L), shape.num_v_heads)
    cfg, ocfg = _cfgs(shape, "bf16", raw, dev)
    H, dk, dv, D = shape.num_v_heads, shape.head_k_dim, shape.head_v_dim, shape.D
    qkv, w = to_dev(v["qkv"], dev), to_dev(v["conv_weight"], dev)
    a, b = to_dev(raw["a"], dev), to_dev(raw["b"], dev)
    conv0, S0 = to_dev(v["conv_state"], dev), to_dev(v["ssm_state"], dev)
    csnap = torch.empty(B, L, D, 3, dtype=torch.bfloat16, device=dev)
    ssnap = torch.empty(B, L, H, dk, dv, device=dev)
    out = torch.empty(B, L, H, dv, device=dev)
    gb.gdn_forward_verify(cfg, B, L, qkv, w, a, b, conv0, S0, csnap, ssnap, out)
    conv_d, S_d = conv0.clone(), S0.clone()
    o1 = torch.empty(B, H, dv, device=dev)
    for t in range(L):
        gb.gdn_forward_decode(cfg, B, qkv[:, :, t].contiguous(), w, a[:, t].contiguous(), b[:, t].contiguous(),
                              conv_d, S_d, o1)
        torch.cuda.synchronize()
        assert np.array_equal(bits(S_d), bits(ssnap[:, t])), f"state snapshot {t}"
        assert np.array_equal(bits(o1), bits(out[:, t])), f"output {t}"
    g_r, b_r = oracle.gate_beta(raw["a"], raw["b"], raw["A_log"], raw["dt_bias"])
    o_r, _, ss_r = oracle.verify(ocfg, f64(v["qkv"]), f64(v["conv_weight"]), g_r, b_r, f64(v["conv_state"]),
                                 v["ssm_state"])
    assert_parity(f64(out), o_r, f64(ssnap[:, L - 1]), ss_r[:, L - 1], what="verify vs oracle")


@pytest.mark.parametrize("variant", [gb.GDN_PREFILL_RESIDENT, gb.GDN_PREFILL_CHUNKED], ids=["resident", "chunked"])
def test_prefill_raw_gates(variant):
    dev = device()
    shape = synth.Shape(2, 4, 128, 64, 4)
    x = synth.varlen_prefill(seed=65, shape=shape, lengths=[70, 0, 3, 129])
    cu = x["cu_seqlens"]
    N, T = len(cu) - 1, int(cu[-1])
    raw = synth.raw_gates(66, (T,), shape.num_v_heads)
    cfg, ocfg = _cfgs(shape, "bf16", raw, dev)
    conv, S = to_dev(x["conv_state"], dev), to_dev(x["ssm_state"], dev)
    out = torch.full((T, shape.num_v_heads, shape.head_v_dim), float("nan"), device=dev)
    ws = torch.empty(max(1, gb.gdn_prefill_workspace_size(cfg, N, T, variant)), dtype=torch.uint8, device=dev)
    gb.gdn_forward_prefill(cfg, N, to_dev(cu, dev), torch.from_numpy(cu), to_dev(x["qkv"], dev),
                           to_dev(x["conv_weight"], dev), to_dev(raw["a"], dev), to_dev(raw["b"], dev), conv, S, out,
                           variant, ws)
    g_r, b_r = oracle.gate_beta(raw["a"], raw["b"], raw["A_log"], raw["dt_bias"])
    o_r, c_r, S_r = oracle.prefill(ocfg, cu, f64(x["qkv"]), f64(x["conv_weight"]), g_r, b_r, f64(x["conv_state"]),
                                   x["ssm_state"])
    torch.cuda.synchronize()
    assert_parity(f64(out), o_r, f64(S), S_r, what="prefill with raw gates")
    assert np.array_equal(f64(conv), c_r)
