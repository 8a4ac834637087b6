"""Prefill over cu_seqlens-packed sequences against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_causal_gb300 import binding as gb
from gated_deltanet_linear_causal_gb300 import synth
from gdn_testutil import Guarded, assert_parity, bits, configs, device, f64, to_dev
from oracle_pool import heads_reference

pytestmark = pytest.mark.gpu

VARIANTS = [gb.GDN_PREFILL_RESIDENT]


def _prefill_dev(cfg, x, dev, variant, io):
    cvt = (lambda a: a) if io == "bf16" else (lambda a: synth.bf16_bits_to_f32(a) if a.dtype == np.uint16 else a)
    cu = x["cu_seqlens"]
    N, T = len(cu) - 1, int(cu[-1])
    H, dv = cfg.num_v_heads, cfg.head_v_dim
    d = dict(cu=to_dev(cu, dev), qkv=to_dev(cvt(x["qkv"]), dev), w=to_dev(cvt(x["conv_weight"]), dev),
             gate=to_dev(x["gate"], dev), beta=to_dev(x["beta"], dev), conv=to_dev(cvt(x["conv_state"]), dev),
             S=to_dev(x["ssm_state"], dev), out=torch.full((T, H, dv), float("nan"), device=dev))
    ws = torch.empty(max(1, gb.gdn_prefill_workspace_size(cfg, N, T, variant)), dtype=torch.uint8, device=dev)
    gb.gdn_forward_prefill(cfg, N, d["cu"], torch.from_numpy(cu), d["qkv"], d["w"], d["gate"], d["beta"], d["conv"],
                           d["S"], d["out"], variant, ws)
    return d


def _oracle_prefill(ocfg, x, seq_index=None):
    return oracle.prefill(ocfg, x["cu_seqlens"], f64(x["qkv"]), f64(x["conv_weight"]), x["gate"], x["beta"],
                          f64(x["conv_state"]), x["ssm_state"], seq_index)


@pytest.mark.parametrize("variant", VARIANTS)
def test_prefill_oracle_scale_f32(variant):
    """B=1, L=64, H_k=2, H_v=4, d=32, K=4, fp32 inputs, zero initial states."""
    dev = device()
    shape = synth.ORACLE_SCALE
    cfg, ocfg = configs(shape, "f32")
    s = synth.oracle_scale(seed=1)
    x = dict(cu_seqlens=np.array([0, 64], np.int32), qkv=s["qkv"][0], conv_weight=s["conv_weight"],
             gate=s["gate"][0], beta=s["beta"][0], conv_state=s["conv_state"], ssm_state=s["ssm_state"])
    d = _prefill_dev(cfg, x, dev, variant, "f32")
    o_r, c_r, S_r = _oracle_prefill(ocfg, x)
    torch.cuda.synchronize()
    assert_parity(f64(d["out"]), o_r, f64(d["S"]), S_r)
    assert np.array_equal(f64(d["conv"]), c_r)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_prefill_varlen_ragged(variant, io):
    """Empty sequences, sequences shorter than the conv window, and ragged tails."""
    dev = device()
    shape = synth.Shape(2, 4, 32, 64, 4)
    cfg, ocfg = configs(shape, io)
    lengths = [0, 1, 2, 3, 17, 40, 0, 5, 130, 1]
    x = synth.varlen_prefill(seed=31, shape=shape, lengths=lengths)
    d = _prefill_dev(cfg, x, dev, variant, io)
    o_r, c_r, S_r = _oracle_prefill(ocfg, x)
    torch.cuda.synchronize()
    assert_parity(f64(d["out"]), o_r, f64(d["S"]), S_r)
    assert np.array_equal(f64(d["conv"]), c_r)


@pytest.mark.parametrize("dk,dv,hk,hv,K", [(64, 64, 1, 1, 4), (128, 32, 2, 8, 2), (256, 64, 1, 2, 4),
                                           (32, 96, 3, 6, 1)])
def test_prefill_head_shapes(dk, dv, hk, hv, K):
    dev = device()
    shape = synth.Shape(hk, hv, dk, dv, K)
    cfg, ocfg = configs(shape, "bf16")
    x = synth.varlen_prefill(seed=dk + dv, shape=shape, lengths=[37, 3, 64])
    d = _prefill_dev(cfg, x, dev, gb.GDN_PREFILL_RESIDENT, "bf16")
    o_r, c_r, S_r = _oracle_prefill(ocfg, x)
    torch.cuda.synchronize()
    assert_parity(f64(d["out"]), o_r, f64(d["S"]), S_r)
    assert np.array_equal(f64(d["conv"]), c_r)


@pytest.mark.parametrize("cut", [40, 37])
def test_prefill_split_equals_whole(cut):
    """Two calls with carried conv and SSM states equal one call.  The kernel works in
    blocks of 8 tokens from each call's start, so a cut on a block boundary (40)
    reproduces the bits of one call and any other cut (37) agrees to rounding."""
    dev = device()
    shape = synth.Shape(2, 4, 64, 64, 4)
    cfg, _ = configs(shape, "bf16")
    x = synth.varlen_prefill(seed=55, shape=shape, lengths=[90])
    whole = _prefill_dev(cfg, x, dev, gb.GDN_PREFILL_RESIDENT, "bf16")
    a = dict(x, cu_seqlens=np.array([0, cut], np.int32), qkv=np.ascontiguousarray(x["qkv"][:, :cut]),
             gate=x["gate"][:cut], beta=x["beta"][:cut])
    da = _prefill_dev(cfg, a, dev, gb.GDN_PREFILL_RESIDENT, "bf16")
    torch.cuda.synchronize()
    b = dict(x, cu_seqlens=np.array([0, 90 - cut], np.int32), qkv=np.ascontiguousarray(x["qkv"][:, cut:]),
             gate=x["gate"][cut:], beta=x["beta"][cut:],
             conv_state=da["conv"].cpu().view(torch.int16).numpy().view(np.uint16),
             ssm_state=da["S"].cpu().numpy())
    db = _prefill_dev(cfg, b, dev, gb.GDN_PREFILL_RESIDENT, "bf16")
    torch.cuda.synchronize()
    out = torch.cat([da["out"], db["out"]])
    assert np.array_equal(bits(db["conv"]), bits(whole["conv"]))
    if cut % 8 == 0:
        assert np.array_equal(bits(out), bits(whole["out"]))
        assert np.array_equal(bits(db["S"]), bits(whole["S"]))
    else:
        assert_parity(f64(out), f64(whole["out"]), f64(db["S"]), f64(whole["S"]), what="split vs whole")


BOTH = [gb.GDN_PREFILL_RESIDENT, gb.GDN_PREFILL_CHUNKED]


@pytest.fixture(scope="module")
def long_ref():
    """The L=8192 workload and the oracle's result for every value head (one spawned
    job per head)."""
    _, ocfg = configs(synth.PRODUCTION, "bf16")
    x = synth.long_prefill(seed=3)
    return x, heads_reference(ocfg, x, [(0, h) for h in range(synth.PRODUCTION.num_v_heads)])


@pytest.fixture(scope="module")
def varlen_ref():
    """The 16-sequence packed workload and the oracle's result for every (sequence, head)."""
    _, ocfg = configs(synth.PRODUCTION, "bf16")
    x = synth.varlen_prefill(seed=4)
    N = len(x["cu_seqlens"]) - 1
    return x, heads_reference(ocfg, x, [(n, h) for n in range(N) for h in range(synth.PRODUCTION.num_v_heads)])


@pytest.mark.parametrize("variant", BOTH, ids=["resident", "chunked"])
def test_prefill_long_production_all_heads(variant, long_ref):
    """B=1, L=8192, H_k=16, H_v=32, d=128, slow decay: the whole layer on the GPU, every
    value head's output and final state against the oracle, and the output buffer's guard
    bands untouched."""
    dev = device()
    shape = synth.PRODUCTION
    cfg, _ = configs(shape, "bf16")
    x, ref = long_ref
    cu = x["cu_seqlens"]
    T = int(cu[-1])
    conv, S = to_dev(x["conv_state"], dev), to_dev(x["ssm_state"], dev)
    out = Guarded((T, shape.num_v_heads, shape.head_v_dim), torch.float32, dev)
    ws = torch.empty(max(1, gb.gdn_prefill_workspace_size(cfg, 1, T, variant)), dtype=torch.uint8, device=dev)
    gb.gdn_forward_prefill(cfg, 1, to_dev(cu, dev), cu, to_dev(x["qkv"], dev), to_dev(x["conv_weight"], dev),
                           to_dev(x["gate"], dev), to_dev(x["beta"], dev), conv, S, out.t, variant, ws)
    torch.cuda.synchronize()
    o, Sg = f64(out.t), f64(S)
    assert np.isfinite(o).all()
    for h in range(shape.num_v_heads):
        o_r, S_r = ref[(0, h)]
        assert_parity(o[:, h], o_r, Sg[0, h], S_r, what=f"head {h}")
    out.check("output")
    tail = f64(x["qkv"][:, -3:])
    assert np.array_equal(f64(conv)[0], tail), "conv state = last K-1 raw inputs"


@pytest.mark.parametrize("variant", BOTH, ids=["resident", "chunked"])
def test_prefill_varlen_production_all(variant, varlen_ref):
    """16 sequences with lengths U{256..2048}, random per-sequence states: every sequence's
    output, final state and conv state for every value head against the oracle."""
    dev = device()
    shape = synth.PRODUCTION
    cfg, _ = configs(shape, "bf16")
    x, ref = varlen_ref
    d = _prefill_dev(cfg, x, dev, variant, "bf16")
    torch.cuda.synchronize()
    out, S = f64(d["out"]), f64(d["S"])
    cu = x["cu_seqlens"]
    for (n, h), (o_r, S_r) in sorted(ref.items()):
        assert_parity(out[cu[n]:cu[n + 1], h], o_r, S[n, h], S_r, what=f"seq {n} head {h}")
    for n in range(len(cu) - 1):
        assert np.array_equal(f64(d["conv"])[n], f64(x["qkv"][:, cu[n + 1] - 3:cu[n + 1]]))


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("hv,dv", [(4, 64), (2, 32), (8, 96)])
def test_prefill_chunked_ragged(io, hv, dv):
    """The tensor-core chunked form (d_k = 128, 64-token chunks): empty sequences,
    sequences shorter than the conv window, chunk-aligned and ragged tails, several
    GQA ratios, every output and state against the oracle."""
    dev = device()
    shape = synth.Shape(2, hv, 128, dv, 4)
    cfg, ocfg = configs(shape, io)
    lengths = [0, 1, 2, 3, 17, 64, 65, 130, 0, 200, 5]
    x = synth.varlen_prefill(seed=70 + hv + dv, shape=shape, lengths=lengths)
    d = _prefill_dev(cfg, x, dev, gb.GDN_PREFILL_CHUNKED, io)
    o_r, c_r, S_r = _oracle_prefill(ocfg, x)
    torch.cuda.synchronize()
    assert_parity(f64(d["out"]), o_r, f64(d["S"]), S_r, what="chunked")
    assert np.array_equal(f64(d["conv"]), c_r)


def test_prefill_chunked_matches_resident():
    """Both prefill forms agree to rounding on the same inputs (fast decay, random states)."""
    dev = device()
    shape = synth.Shape(4, 8, 128, 128, 4)
    cfg, _ = configs(shape, "bf16")
    x = synth.varlen_prefill(seed=81, shape=shape, lengths=[300, 1, 129])
    r = _prefill_dev(cfg, x, dev, gb.GDN_PREFILL_RESIDENT, "bf16")
    c = _prefill_dev(cfg, x, dev, gb.GDN_PREFILL_CHUNKED, "bf16")
    torch.cuda.synchronize()
    assert_parity(f64(c["out"]), f64(r["out"]), f64(c["S"]), f64(r["S"]), what="chunked vs resident")
    assert torch.equal(c["conv"], r["conv"])


def test_prefill_chunked_rejects_other_head_sizes():
    dev = device()
    shape = synth.Shape(2, 4, 64, 64, 4)
    cfg, _ = configs(shape, "bf16")
    x = synth.varlen_prefill(seed=5, shape=shape, lengths=[10])
    with pytest.raises(gb.GdnError) as e:
        _prefill_dev(cfg, x, dev, gb.GDN_PREFILL_CHUNKED, "bf16")
    assert e.value.status == 8


def test_prefill_empty_is_noop():
    dev = device()
    cfg, _ = configs(synth.ORACLE_SCALE, "f32")
    z = torch.zeros(64, device=dev)
    conv = torch.zeros(2, cfg.D, 3, device=dev)
    S = torch.ones(2, 4, 32, 32, device=dev)
    gb.gdn_forward_prefill(cfg, 2, torch.zeros(3, dtype=torch.int32, device=dev), np.zeros(3, np.int32), z, z, z, z,
                           conv, S, z, gb.GDN_PREFILL_RESIDENT, None)
    torch.cuda.synchronize()
    assert bool((S == 1).all())


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_prefill_resident_without_l2norm(io):
    """use_qk_l2norm = 0: only the 1/sqrt(d_k) scale; short sequences keep the un-normalised
    recurrence (|k|^2 of tens) within fp32 range."""
    dev = device()
    shape = synth.Shape(2, 4, 64, 32, 4)
    cfg, ocfg = configs(shape, io, use_l2=False)
    x = synth.varlen_prefill(seed=95, shape=shape, lengths=[3, 0, 6, 1])
    d = _prefill_dev(cfg, x, dev, gb.GDN_PREFILL_RESIDENT, io)
    o_r, c_r, S_r = _oracle_prefill(ocfg, x)
    torch.cuda.synchronize()
    assert_parity(f64(d["out"]), o_r, f64(d["S"]), S_r, what="resident, no L2 norm")


def test_prefill_chunked_requires_l2norm():
    dev = device()
    shape = synth.Shape(2, 4, 128, 64, 4)
    cfg, _ = configs(shape, "bf16", use_l2=False)
    x = synth.varlen_prefill(seed=96, shape=shape, lengths=[10])
    with pytest.raises(gb.GdnError) as e:
        _prefill_dev(cfg, x, dev, gb.GDN_PREFILL_CHUNKED, "bf16")
    assert e.value.status == 8


@pytest.mark.parametrize("K,misaligned", [(1, False), (2, False), (3, False), (4, True), (3, True)])
def test_prefill_chunked_conv_widths(K, misaligned):
    """The chunked form's staged conv: widths below 4 (weight rows of K taps) and a
    conv-weight buffer that starts off a 16-byte boundary (weights then load without the
    16-byte copies), against the oracle."""
    dev = device()
    shape = synth.Shape(2, 4, 128, 64, K)
    cfg, ocfg = configs(shape, "bf16")
    x = synth.varlen_prefill(seed=140 + K + 7 * misaligned, shape=shape, lengths=[70, 2, 1, 129])
    cu = x["cu_seqlens"]
    N, T = len(cu) - 1, int(cu[-1])
    w = to_dev(x["conv_weight"], dev)
    if misaligned:
        buf = torch.empty(w.numel() + 1, dtype=w.dtype, device=dev)
        buf[1:].copy_(w.reshape(-1))
        w = buf[1:].view(w.shape)
        assert w.data_ptr() % 16 != 0
    d = dict(qkv=to_dev(x["qkv"], dev), gate=to_dev(x["gate"], dev), beta=to_dev(x["beta"], dev),
             conv=to_dev(x["conv_state"], dev), S=to_dev(x["ssm_state"], dev),
             out=torch.full((T, shape.num_v_heads, shape.head_v_dim), float("nan"), device=dev))
    var = gb.GDN_PREFILL_CHUNKED
    ws = torch.empty(max(1, gb.gdn_prefill_workspace_size(cfg, N, T, var)), dtype=torch.uint8, device=dev)
    gb.gdn_forward_prefill(cfg, N, to_dev(cu, dev), torch.from_numpy(cu), d["qkv"], w, d["gate"], d["beta"], d["conv"],
                           d["S"], d["out"], var, ws)
    o_r, c_r, S_r = _oracle_prefill(ocfg, x)
    torch.cuda.synchronize()
    assert_parity(f64(d["out"]), o_r, f64(d["S"]), S_r, what=f"chunked K={K}")
    assert np.array_equal(f64(d["conv"]), c_r)


@pytest.mark.parametrize("cut", [64, 37])
def test_prefill_chunked_split_equals_whole(cut):
    """Two chunked calls with carried conv and SSM states agree with one call: the second
    call's first chunk takes its conv window's head from the carried conv state."""
    dev = device()
    shape = synth.Shape(2, 4, 128, 64, 4)
    cfg, _ = configs(shape, "bf16")
    x = synth.varlen_prefill(seed=57, shape=shape, lengths=[150])
    var = gb.GDN_PREFILL_CHUNKED
    whole = _prefill_dev(cfg, x, dev, var, "bf16")
    a = dict(x, cu_seqlens=np.array([0, cut], np.int32), qkv=np.ascontiguousarray(x["qkv"][:, :cut]),
             gate=x["gate"][:cut], beta=x["beta"][:cut])
    da = _prefill_dev(cfg, a, dev, var, "bf16")
    torch.cuda.synchronize()
    b = dict(x, cu_seqlens=np.array([0, 150 - cut], np.int32), qkv=np.ascontiguousarray(x["qkv"][:, cut:]),
             gate=x["gate"][cut:], beta=x["beta"][cut:],
             conv_state=da["conv"].cpu().view(torch.int16).numpy().view(np.uint16),
             ssm_state=da["S"].cpu().numpy())
    db = _prefill_dev(cfg, b, dev, var, "bf16")
    torch.cuda.synchronize()
    out = torch.cat([da["out"], db["out"]])
    assert np.array_equal(bits(db["conv"]), bits(whole["conv"]))
    assert_parity(f64(out), f64(whole["out"]), f64(db["S"]), f64(whole["S"]), what="chunked split vs whole")
