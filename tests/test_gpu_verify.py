"""MTP verify (per-token snapshots) and commit (rollback to the accepted prefix)."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_causal_gb300 import binding as gb
from gated_deltanet_linear_causal_gb300 import synth
from gdn_testutil import assert_parity, bits, configs, device, f64, to_dev

pytestmark = pytest.mark.gpu


def _verify(shape, io, batch, L, seed):
    dev = device()
    cfg, ocfg = configs(shape, io)
    v = synth.verify_block(seed, batch, L, shape)
    cvt = (lambda a: a) if io == "bf16" else synth.bf16_bits_to_f32
    H, dk, dv, D, K = shape.num_v_heads, shape.head_k_dim, shape.head_v_dim, shape.D, shape.conv_kernel
    x = dict(qkv=to_dev(cvt(v["qkv"]), dev), w=to_dev(cvt(v["conv_weight"]), dev), gate=to_dev(v["gate"], dev),
             beta=to_dev(v["beta"], dev), conv=to_dev(cvt(v["conv_state"]), dev), S=to_dev(v["ssm_state"], dev))
    csnap = torch.empty(batch, L, D, K - 1, dtype=cfg.torch_dtype, device=dev)
    ssnap = torch.empty(batch, L, H, dk, dv, device=dev)
    out = torch.empty(batch, L, H, dv, device=dev)
    gb.gdn_forward_verify(cfg, batch, L, x["qkv"], x["w"], x["gate"], x["beta"], x["conv"], x["S"], csnap, ssnap, out)
    return cfg, ocfg, v, x, csnap, ssnap, out


def test_verify_production_b32_l4_and_commit():
    """B=32 sequences, L=4 draft tokens: outputs and every snapshot against the oracle,
    then commit a seeded accepted length per sequence."""
    shape = synth.PRODUCTION
    cfg, ocfg, v, x, csnap, ssnap, out = _verify(shape, "bf16", 32, 4, seed=5)
    S_prior = x["S"].clone()
    conv_prior = x["conv"].clone()
    o_r, cs_r, ss_r = oracle.verify(ocfg, f64(v["qkv"]), f64(v["conv_weight"]), v["gate"], v["beta"],
                                    f64(v["conv_state"]), v["ssm_state"])
    torch.cuda.synchronize()
    assert_parity(f64(out), o_r, what="verify outputs")
    for t in range(4):
        assert_parity(f64(out[:, t]), o_r[:, t], f64(ssnap[:, t]), ss_r[:, t], what=f"snapshot {t}")
    assert np.array_equal(f64(csnap), cs_r), "conv snapshots are exact raw inputs"
    # the live states are read only
    assert torch.equal(x["S"], S_prior) and torch.equal(x["conv"], conv_prior)

    acc = v["accepted"]
    status = torch.zeros(1, dtype=torch.int32, device=x["S"].device)
    gb.gdn_verify_commit(cfg, 32, 4, to_dev(acc, x["S"].device), csnap, ssnap, x["conv"], x["S"], status)
    conv_r, S_r = oracle.commit(f64(v["conv_state"]), v["ssm_state"], cs_r, ss_r, acc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for b in range(32):
        if acc[b] == 0:
            assert torch.equal(x["S"][b], S_prior[b]) and torch.equal(x["conv"][b], conv_prior[b])
        else:
            assert torch.equal(x["S"][b], ssnap[b, acc[b] - 1])
            assert_parity(f64(out[b, acc[b] - 1]), o_r[b, acc[b] - 1], f64(x["S"][b]), S_r[b], what=f"commit b={b}")
    assert np.array_equal(f64(x["conv"]), conv_r)


@pytest.mark.parametrize("io,dk,dv", [("bf16", 128, 64), ("f32", 32, 64), ("bf16", 64, 64), ("f32", 256, 64),
                                      ("bf16", 128, 128), ("f32", 64, 128), ("bf16", 128, 256)])
def test_verify_snapshot_bitwise_equals_decode(io, dk, dv):
    """Snapshot t equals, bit for bit, the states t+1 decode calls leave (the verify
    block and single steps run the same per-token arithmetic)."""
    shape = synth.Shape(2, 4, dk, dv, 4)
    L, batch = 5, 3
    cfg, ocfg, v, x, csnap, ssnap, out = _verify(shape, io, batch, L, seed=dk)
    dev = x["S"].device
    conv, S = x["conv"].clone(), x["S"].clone()
    o1 = torch.empty(batch, shape.num_v_heads, shape.head_v_dim, device=dev)
    for t in range(L):
        gb.gdn_forward_decode(cfg, batch, x["qkv"][:, :, t].contiguous(), x["w"], x["gate"][:, t].contiguous(),
                              x["beta"][:, t].contiguous(), conv, S, o1)
        torch.cuda.synchronize()
        assert np.array_equal(bits(S), bits(ssnap[:, t])), f"ssm snapshot {t}"
        assert np.array_equal(bits(conv), bits(csnap[:, t])), f"conv snapshot {t}"
        assert np.array_equal(bits(o1), bits(out[:, t])), f"output {t}"


def test_commit_rejects_out_of_range_accepted():
    shape = synth.Shape(1, 2, 32, 32, 4)
    cfg, ocfg, v, x, csnap, ssnap, out = _verify(shape, "f32", 4, 3, seed=9)
    dev = x["S"].device
    S0, c0 = x["S"].clone(), x["conv"].clone()
    acc = torch.tensor([3, -1, 4, 1], dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    gb.gdn_verify_commit(cfg, 4, 3, acc, csnap, ssnap, x["conv"], x["S"], status)
    torch.cuda.synchronize()
    assert int(status.item()) == gb.GDN_ERR_RANGE
    assert torch.equal(x["S"][1], S0[1]) and torch.equal(x["S"][2], S0[2])
    assert torch.equal(x["conv"][1], c0[1]) and torch.equal(x["conv"][2], c0[2])
    assert torch.equal(x["S"][0], ssnap[0, 2]) and torch.equal(x["S"][3], ssnap[3, 0])
    assert torch.equal(x["conv"][0], csnap[0, 2])


@pytest.mark.parametrize("L", [1, 2, 16])
def test_verify_block_lengths(L):
    shape = synth.Shape(2, 4, 64, 64, 4)
    cfg, ocfg, v, x, csnap, ssnap, out = _verify(shape, "bf16", 2, L, seed=100 + L)
    o_r, cs_r, ss_r = oracle.verify(ocfg, f64(v["qkv"]), f64(v["conv_weight"]), v["gate"], v["beta"],
                                    f64(v["conv_state"]), v["ssm_state"])
    torch.cuda.synchronize()
    assert_parity(f64(out), o_r, f64(ssnap[:, -1]), ss_r[:, -1], what=f"L={L}")
    assert np.array_equal(f64(csnap), cs_r)


def test_verify_without_l2norm_stream_kernel():
    """use_qk_l2norm = 0 on the streaming kernel's shape (d = 128), L = 2: outputs and
    snapshots against the oracle."""
    dev = device()
    shape = synth.Shape(2, 4, 128, 128, 4)
    cfg, ocfg = configs(shape, "bf16", use_l2=False)
    B, L = 3, 2
    v = synth.verify_block(97, B, L, shape)
    H, dk, dv, D = shape.num_v_heads, shape.head_k_dim, shape.head_v_dim, shape.D
    csnap = torch.empty(B, L, D, 3, dtype=torch.bfloat16, device=dev)
    ssnap = torch.empty(B, L, H, dk, dv, device=dev)
    out = torch.empty(B, L, H, dv, device=dev)
    gb.gdn_forward_verify(cfg, B, L, to_dev(v["qkv"], dev), to_dev(v["conv_weight"], dev), to_dev(v["gate"], dev),
                          to_dev(v["beta"], dev), to_dev(v["conv_state"], dev), to_dev(v["ssm_state"], dev), csnap,
                          ssnap, out)
    o_r, cs_r, ss_r = oracle.verify(ocfg, f64(v["qkv"]), f64(v["conv_weight"]), v["gate"], v["beta"],
                                    f64(v["conv_state"]), v["ssm_state"])
    torch.cuda.synchronize()
    for t in range(L):
        assert_parity(f64(out[:, t]), o_r[:, t], f64(ssnap[:, t]), ss_r[:, t], what=f"snapshot {t}")
