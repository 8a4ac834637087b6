"""Gated RMSNorm of the layer output (section 2): the standalone kernel over rows of
head_v_dim, and the decode kernel and both prefill forms with the norm fused into
their output epilogues, against the fp64 oracle (oracle.gated_rmsnorm after
oracle.decode / oracle.prefill).

Tolerance of y: the standalone norm gets exact inputs, so its error is the fp32
arithmetic plus, for a bf16 output, one rounding to bf16 (relative 2^-9):
|dy| <= 2^-8 |y_ref| + 1e-6 RMS(y_ref) (fp32 output: 1e-5 |y_ref| + 1e-6 RMS).  The
fused decode also carries the layer output's own error, |do| <= e = 2e-3 RMS(o):
to first order y_j = w_j s_j o_j / rms moves by w_j s_j (do_j - o_j drms/rms) / rms
with |drms| <= e, so each element is held to
    |dy_j| <= 2^-8 |y_ref_j| + |w_j silu(z_j)| (e / rms) (1 + |o_j| / rms),
rms the row's RMS of the oracle output; and to one bf16 step against the unfused
GPU path (decode, then the standalone norm), bitwise for the states."""
import numpy as np
import pytest
import scipy.special
import torch

import oracle
from gated_deltanet_linear_causal_gb300 import binding as gb
from gated_deltanet_linear_causal_gb300 import synth
from gdn_testutil import O_TOL, Guarded, bits, configs, device, f64, to_dev

pytestmark = pytest.mark.gpu


def _check_y(y, y_ref, rel, what):
    y, y_ref = np.asarray(y, np.float64), np.asarray(y_ref, np.float64)
    rms = np.sqrt(np.mean(y_ref ** 2))
    bad = np.abs(y - y_ref) > rel * np.abs(y_ref) + 1e-6 * rms
    assert not bad.any(), f"{what}: {bad.sum()} elements off, worst {np.max(np.abs(y - y_ref) / (np.abs(y_ref) + rms)):.3g}"


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("dv", [32, 96, 128])
def test_gated_rmsnorm_standalone(io, dv):
    dev = device()
    shape = synth.Shape(1, 2, 32, dv, 4)
    cfg, _ = configs(shape, io)
    d = synth.Draw(90 + dv)
    rows = 37
    o = d.f32("o", (rows, dv), 0.0, 2.0)
    z = d.bf16("z", (rows, dv), 0.0, 1.5)
    zin = z if io == "bf16" else synth.bf16_bits_to_f32(z)
    w = d.f32("w", (dv,), 1.0, 0.3)
    y = torch.empty(rows, dv, dtype=cfg.torch_dtype, device=dev)
    gb.gdn_gated_rmsnorm(cfg, rows, to_dev(o, dev), to_dev(zin, dev), to_dev(w, dev), 1e-6, y)
    y_ref = oracle.gated_rmsnorm(o, f64(zin), w, 1e-6)
    torch.cuda.synchronize()
    _check_y(f64(y), y_ref, 2.0 ** -8 if io == "bf16" else 1e-5, f"standalone {io} dv={dv}")


def test_decode_gated_fused_production():
    dev = device()
    shape, B, steps = synth.PRODUCTION, 8, 3
    H, dv = shape.num_v_heads, shape.head_v_dim
    cfg, ocfg = configs(shape, "bf16")
    st = synth.decode_state(91, B, shape)
    d = synth.Draw(92)
    w_n = to_dev(d.f32("norm_w", (dv,), 1.0, 0.3), dev)
    w = to_dev(st["conv_weight"], dev)
    conv_f, S_f = to_dev(st["conv_state"], dev), to_dev(st["ssm_state"], dev)   # fused path
    conv_u, S_u = conv_f.clone(), S_f.clone()                                      # unfused GPU path
    conv_r, S_r = f64(st["conv_state"]), st["ssm_state"].astype(np.float64)        # oracle
    y = torch.empty(B, H, dv, dtype=torch.bfloat16, device=dev)
    y2 = torch.empty_like(y)
    out = torch.empty(B, H, dv, device=dev)
    for s in range(steps):
        x = synth.decode_step(91, s, B, shape)
        z = d.bf16(f"z{s}", (B, H, dv), 0.0, 1.5)
        qkv, g, b, zd = to_dev(x["qkv"], dev), to_dev(x["gate"], dev), to_dev(x["beta"], dev), to_dev(z, dev)
        gb.gdn_forward_decode_gated(cfg, B, qkv, w, g, b, conv_f, S_f, zd, w_n, 1e-6, y)
        gb.gdn_forward_decode(cfg, B, qkv, w, g, b, conv_u, S_u, out)
        gb.gdn_gated_rmsnorm(cfg, B * H, out, zd, w_n, 1e-6, y2)
        o_r, conv_r, S_r = oracle.decode(ocfg, f64(x["qkv"]), f64(st["conv_weight"]), x["gate"], x["beta"], conv_r,
                                         S_r)
        y_ref = oracle.gated_rmsnorm(o_r, f64(z), f64(w_n), 1e-6)
        torch.cuda.synchronize()
        assert np.array_equal(bits(S_f), bits(S_u)) and np.array_equal(bits(conv_f), bits(conv_u)), "states"
        _check_y(f64(y), f64(y2), 2.0 ** -7, f"step {s}: fused vs decode + norm")
        e_abs = O_TOL * np.sqrt(np.mean(o_r ** 2))
        rms = np.sqrt(np.mean(o_r ** 2, axis=-1, keepdims=True) + 1e-6)
        zf = f64(z)
        gate = np.abs(f64(w_n) * zf * scipy.special.expit(zf))
        bound = 2.0 ** -8 * np.abs(y_ref) + gate * (e_abs / rms) * (1.0 + np.abs(o_r) / rms)
        err = np.abs(f64(y) - y_ref)
        assert (err <= bound).all(), f"step {s}: worst err/bound {np.max(err / bound):.3g}"


def test_decode_gated_rejects_other_value_dims():
    dev = device()
    shape = synth.Shape(2, 4, 128, 64, 4)
    cfg, _ = configs(shape, "bf16")
    t = lambda n, dt=torch.float32: torch.zeros(n, dtype=dt, device=dev)
    B, D = 2, shape.D
    with pytest.raises(gb.GdnError) as e:
        gb.gdn_forward_decode_gated(cfg, B, t(B * D, torch.bfloat16), t(D * 4, torch.bfloat16), t(B * 4), t(B * 4),
                                    t(B * D * 3, torch.bfloat16), t(B * 4 * 128 * 64), t(B * 4 * 64, torch.bfloat16),
                                    t(64), 1e-6, t(B * 4 * 64, torch.bfloat16))
    assert e.value.status == 8


def _oracle_bound(y_ref, o_r, zf, w):
    """First-order bound of the normalised output from the layer's own bound |do| <= 2e-3 RMS(o)."""
    e_abs = O_TOL * np.sqrt(np.mean(o_r ** 2))
    rms = np.sqrt(np.mean(o_r ** 2, axis=-1, keepdims=True) + 1e-6)
    gate = np.abs(w * zf * scipy.special.expit(zf))
    return 2.0 ** -8 * np.abs(y_ref) + gate * (e_abs / rms) * (1.0 + np.abs(o_r) / rms)


def _prefill_gated_vs_unfused(shape, io, variant, lengths, seed):
    """Fused prefill + norm against (a) the plain prefill then the standalone norm on the GPU
    (states bitwise, y to one bf16 step) and (b) the oracle (first-order bound)."""
    dev = device()
    cfg, ocfg = configs(shape, io)
    H, dv = shape.num_v_heads, shape.head_v_dim
    x = synth.varlen_prefill(seed=seed, shape=shape, lengths=lengths)
    cvt = (lambda a: a) if io == "bf16" else (lambda a: synth.bf16_bits_to_f32(a) if a.dtype == np.uint16 else a)
    cu = x["cu_seqlens"]
    N, T = len(cu) - 1, int(cu[-1])
    d = synth.Draw(seed + 1)
    z = cvt(d.bf16("z", (T, H, dv), 0.0, 1.5))
    w_n = d.f32("norm_w", (dv,), 1.0, 0.3)
    args = dict(cu=to_dev(cu, dev), qkv=to_dev(cvt(x["qkv"]), dev), w=to_dev(cvt(x["conv_weight"]), dev),
                gate=to_dev(x["gate"], dev), beta=to_dev(x["beta"], dev))
    ws = torch.empty(max(1, gb.gdn_prefill_workspace_size(cfg, N, T, variant)), dtype=torch.uint8, device=dev)
    conv_f, S_f = to_dev(cvt(x["conv_state"]), dev), to_dev(x["ssm_state"], dev)
    conv_u, S_u = conv_f.clone(), S_f.clone()
    y = Guarded((T, H, dv), cfg.torch_dtype, dev)
    gb.gdn_forward_prefill_gated(cfg, N, args["cu"], cu, args["qkv"], args["w"], args["gate"], args["beta"], conv_f,
                                 S_f, to_dev(z, dev), to_dev(w_n, dev), 1e-6, y.t, variant, ws)
    out = torch.empty(T, H, dv, device=dev)
    y2 = torch.empty(T, H, dv, dtype=cfg.torch_dtype, device=dev)
    gb.gdn_forward_prefill(cfg, N, args["cu"], cu, args["qkv"], args["w"], args["gate"], args["beta"], conv_u, S_u,
                           out, variant, ws)
    gb.gdn_gated_rmsnorm(cfg, T * H, out, to_dev(z, dev), to_dev(w_n, dev), 1e-6, y2)
    o_r, _, _ = oracle.prefill(ocfg, cu, f64(cvt(x["qkv"])), f64(cvt(x["conv_weight"])), x["gate"], x["beta"],
                               f64(cvt(x["conv_state"])), x["ssm_state"])
    torch.cuda.synchronize()
    y.check("y")
    assert np.array_equal(bits(S_f), bits(S_u)) and np.array_equal(bits(conv_f), bits(conv_u)), "states"
    _check_y(f64(y.t), f64(y2), 2.0 ** -7 if io == "bf16" else 1e-5, "fused vs prefill + norm")
    zf = f64(z)
    y_ref = oracle.gated_rmsnorm(o_r, zf, w_n, 1e-6)
    bound = _oracle_bound(y_ref, o_r, zf, w_n.astype(np.float64))
    err = np.abs(f64(y.t) - y_ref)
    assert (err <= bound).all(), f"against the oracle: worst err/bound {np.max(err / bound):.3g}"


@pytest.mark.parametrize("variant,shape,io", [
    (gb.GDN_PREFILL_CHUNKED, synth.Shape(2, 4, 128, 128, 4), "bf16"),
    (gb.GDN_PREFILL_CHUNKED, synth.Shape(2, 4, 128, 64, 4), "f32"),
    (gb.GDN_PREFILL_CHUNKED, synth.Shape(2, 2, 128, 96, 4), "bf16"),
    (gb.GDN_PREFILL_RESIDENT, synth.Shape(2, 4, 128, 128, 4), "bf16"),
    (gb.GDN_PREFILL_RESIDENT, synth.Shape(2, 4, 64, 64, 4), "f32"),
    (gb.GDN_PREFILL_RESIDENT, synth.Shape(1, 2, 32, 32, 4), "bf16"),
], ids=["chunked-128", "chunked-64-f32", "chunked-96", "resident-128", "resident-64-f32", "resident-32"])
def test_prefill_gated_fused(variant, shape, io):
    """Ragged packed sequences: several chunks with a tail, one exact chunk, one token, an
    empty one, a short one."""
    _prefill_gated_vs_unfused(shape, io, variant, [150, 64, 1, 0, 37], seed=170 + shape.head_v_dim)


@pytest.mark.parametrize("variant", [gb.GDN_PREFILL_CHUNKED, gb.GDN_PREFILL_RESIDENT], ids=["chunked", "resident"])
def test_prefill_gated_fused_production_heads(variant):
    """H_k=16, H_v=32, d=128 over 1024 tokens: every head's normalised output."""
    _prefill_gated_vs_unfused(synth.PRODUCTION, "bf16", variant, [1024], seed=180)


def test_prefill_gated_rejects_wide_value_heads():
    dev = device()
    shape = synth.Shape(1, 1, 64, 256, 4)   # resident clusters of dv/16 = 16 CTAs: more than 8
    cfg, _ = configs(shape, "bf16")
    T, D = 4, shape.D
    t = lambda n, dt=torch.float32: torch.zeros(n, dtype=dt, device=dev)
    cu = np.array([0, T], np.int32)
    ws = torch.empty(gb.gdn_prefill_workspace_size(cfg, 1, T), dtype=torch.uint8, device=dev)
    with pytest.raises(gb.GdnError) as e:
        gb.gdn_forward_prefill_gated(cfg, 1, to_dev(cu, dev), cu, t(D * T, torch.bfloat16), t(D * 4, torch.bfloat16),
                                     t(T), t(T), t(D * 3, torch.bfloat16), t(64 * 256), t(T * 256, torch.bfloat16),
                                     t(256), 1e-6, t(T * 256, torch.bfloat16), gb.GDN_PREFILL_RESIDENT, ws)
    assert e.value.status == 8
