"""Decode (L = 1, states in place) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_causal_gb300 import binding as gb
from gated_deltanet_linear_causal_gb300 import synth
from gdn_testutil import Guarded, assert_parity, configs, device, f64, to_dev

pytestmark = pytest.mark.gpu


def _run_decode_steps(shape, io, batch, steps, seed, use_l2=True, conv_kernel=None):
    if conv_kernel is not None:
        shape = synth.Shape(shape.num_k_heads, shape.num_v_heads, shape.head_k_dim, shape.head_v_dim, conv_kernel)
    dev = device()
    cfg, ocfg = configs(shape, io, use_l2)
    st = synth.decode_state(seed, batch, shape)
    conv_w = st["conv_weight"] if io == "bf16" else synth.bf16_bits_to_f32(st["conv_weight"])
    conv0 = st["conv_state"] if io == "bf16" else synth.bf16_bits_to_f32(st["conv_state"])
    w_d, conv_d, S_d = to_dev(conv_w, dev), to_dev(conv0, dev), to_dev(st["ssm_state"], dev)
    conv_r, S_r = f64(conv0), st["ssm_state"].astype(np.float64)
    out = torch.empty(batch, shape.num_v_heads, shape.head_v_dim, device=dev)
    for step in range(steps):
        d = synth.decode_step(seed, step, batch, shape)
        qkv = d["qkv"] if io == "bf16" else synth.bf16_bits_to_f32(d["qkv"])
        gb.gdn_forward_decode(cfg, batch, to_dev(qkv, dev), w_d, to_dev(d["gate"], dev), to_dev(d["beta"], dev),
                              conv_d, S_d, out)
        o_r, conv_r, S_r = oracle.decode(ocfg, f64(qkv), f64(conv_w), d["gate"], d["beta"], conv_r, S_r)
        torch.cuda.synchronize()
        assert_parity(f64(out), o_r, what=f"step {step} output")
    assert_parity(f64(out), o_r, f64(S_d), S_r, what="final")
    assert np.array_equal(f64(conv_d), conv_r), "conv state must be the exact raw inputs"


def test_decode_oracle_scale_f32():
    _run_decode_steps(synth.ORACLE_SCALE, "f32", batch=3, steps=8, seed=21)


def test_decode_production_b64_bf16():
    """The B=64, H_k=16, H_v=32, d=128 decode workload, three consecutive steps, every sequence checked."""
    _run_decode_steps(synth.PRODUCTION, "bf16", batch=64, steps=3, seed=2)


def test_decode_production_256_steps_drift():
    """The decode workload as timed: B=64, 256 consecutive steps on the same carried states.
    Four sequences (every head) follow the oracle step by step: their outputs are compared at
    every step and their fp32 states every 32 steps, so drift of the carried state over a long
    decode run would show; the other sequences run alongside as in the bench."""
    dev = device()
    shape, B, steps, watch = synth.PRODUCTION, 64, 256, [0, 21, 42, 63]
    cfg, ocfg = configs(shape, "bf16")
    st = synth.decode_state(2, B, shape)
    w_d, conv_d, S_d = to_dev(st["conv_weight"], dev), to_dev(st["conv_state"], dev), to_dev(st["ssm_state"], dev)
    w64 = f64(st["conv_weight"])
    conv_r, S_r = f64(st["conv_state"])[watch], st["ssm_state"][watch].astype(np.float64)
    out = Guarded((B, shape.num_v_heads, shape.head_v_dim), torch.float32, dev)
    worst = 0.0
    for step in range(steps):
        d = synth.decode_step(2, step, B, shape)
        gb.gdn_forward_decode(cfg, B, to_dev(d["qkv"], dev), w_d, to_dev(d["gate"], dev), to_dev(d["beta"], dev),
                              conv_d, S_d, out.t)
        o_r, conv_r, S_r = oracle.decode(ocfg, f64(d["qkv"][watch]), w64, d["gate"][watch], d["beta"][watch],
                                         conv_r, S_r)
        o_g = f64(out.t[watch])
        assert_parity(o_g, o_r, what=f"step {step} output")
        if (step + 1) % 32 == 0:
            S_g = f64(S_d[watch])
            assert_parity(o_g, o_r, S_g, S_r, what=f"step {step} state")
            worst = max(worst, float(np.linalg.norm(S_g - S_r) / np.linalg.norm(S_r)))
    out.check("output")
    assert np.array_equal(f64(conv_d[watch]), conv_r)
    assert worst <= 1e-4


@pytest.mark.parametrize("dk,dv,hk,hv", [(32, 32, 1, 1), (64, 64, 2, 2), (64, 96, 2, 8), (128, 64, 4, 16),
                                         (256, 128, 1, 2), (32, 256, 2, 4),
                                         # shapes of the persistent bulk-copy kernel (dk 64/128, dv % 128 == 0)
                                         (64, 128, 2, 4), (128, 256, 2, 4), (128, 128, 1, 4), (64, 384, 3, 3)])
def test_decode_head_shapes(dk, dv, hk, hv):
    _run_decode_steps(synth.Shape(hk, hv, dk, dv, 4), "bf16", batch=5, steps=3, seed=dk + dv + hv)


@pytest.mark.parametrize("K", [1, 2, 3, 8])
def test_decode_conv_widths(K):
    _run_decode_steps(synth.Shape(2, 4, 32, 32, K), "f32", batch=2, steps=K + 2, seed=40 + K, conv_kernel=K)


@pytest.mark.parametrize("K", [1, 3])
def test_decode_conv_widths_bulk_copy_kernel(K):
    _run_decode_steps(synth.Shape(2, 4, 128, 128, K), "bf16", batch=3, steps=K + 2, seed=50 + K, conv_kernel=K)


def test_decode_without_l2norm():
    _run_decode_steps(synth.Shape(2, 4, 64, 32, 4), "f32", batch=2, steps=3, seed=77, use_l2=False)


def test_decode_batch_zero_is_noop():
    dev = device()
    cfg, _ = configs(synth.ORACLE_SCALE, "f32")
    gb.gdn_forward_decode(cfg, 0, *[torch.empty(16, device=dev)] * 7)


def test_decode_back_to_back_launches():
    """Consecutive decode steps launched without any host synchronisation on the same state
    buffers (the streaming kernel overlaps consecutive launches and must still read each
    step's states only after the previous step has written them), with a verify call in the
    middle reading the live states; everything against the oracle at the end."""
    dev = device()
    shape, B, steps = synth.PRODUCTION, 8, 12
    cfg, ocfg = configs(shape, "bf16")
    st = synth.decode_state(98, B, shape)
    w = to_dev(st["conv_weight"], dev)
    conv_d, S_d = to_dev(st["conv_state"], dev), to_dev(st["ssm_state"], dev)
    xs = [synth.decode_step(98, s, B, shape) for s in range(steps)]
    qkv = [to_dev(x["qkv"], dev) for x in xs]
    g = [to_dev(x["gate"], dev) for x in xs]
    b = [to_dev(x["beta"], dev) for x in xs]
    outs = [torch.empty(B, shape.num_v_heads, shape.head_v_dim, device=dev) for _ in range(steps)]
    half = steps // 2
    H, dk, dv, D = shape.num_v_heads, shape.head_k_dim, shape.head_v_dim, shape.D
    csnap = torch.empty(B, 1, D, 3, dtype=torch.bfloat16, device=dev)
    ssnap = torch.empty(B, 1, H, dk, dv, device=dev)
    vout = torch.empty(B, 1, H, dv, device=dev)
    torch.cuda.synchronize()
    for s in range(steps):
        if s == half:  # verify one token of step `half` from the live states, between two decodes
            gb.gdn_forward_verify(cfg, B, 1, qkv[s].view(B, D, 1), w, g[s].view(B, 1, H), b[s].view(B, 1, H),
                                  conv_d, S_d, csnap, ssnap, vout)
        gb.gdn_forward_decode(cfg, B, qkv[s], w, g[s], b[s], conv_d, S_d, outs[s])
    torch.cuda.synchronize()
    conv_r, S_r = f64(st["conv_state"]), st["ssm_state"].astype(np.float64)
    for s in range(steps):
        o_r, conv_r, S_r = oracle.decode(ocfg, f64(xs[s]["qkv"]), f64(st["conv_weight"]), xs[s]["gate"],
                                         xs[s]["beta"], conv_r, S_r)
        assert_parity(f64(outs[s]), o_r, what=f"step {s}")
        if s == half:
            assert_parity(f64(vout[:, 0]), o_r, f64(ssnap[:, 0]), S_r, what="verify between decodes")
    assert_parity(f64(outs[-1]), o_r, f64(S_d), S_r, what="final")
    assert np.array_equal(f64(conv_d), conv_r)
