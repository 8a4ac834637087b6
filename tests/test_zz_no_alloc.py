"""gdn_forward_prefill_noalloc: the prefill entry point that allocates nothing.

It exists for callers that cannot call cudaMalloc: a host framework that owns all
device memory through its own pool, or a serving loop that may not touch the
allocator (cudaMalloc can synchronise the device).  It runs the resident prefill
with its workspace in a fixed device array inside the library.  These tests call
it through the C ABI and compare it with gdn_forward_prefill, whose workspace
comes from the caller, on two calls in a row with different inputs: both run the
same kernels on the same inputs, so the results must agree bit for bit.  (This file
sorts last so that a stop-at-first-failure run has already run every other test.)
"""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_causal_gb300 import binding as gb
from gated_deltanet_linear_causal_gb300 import synth
from gdn_testutil import assert_parity, bits, configs, device, f64, to_dev

pytestmark = pytest.mark.gpu


def _inputs(x, dev):
    return dict(cu=to_dev(x["cu_seqlens"], dev), qkv=to_dev(x["qkv"], dev), w=to_dev(x["conv_weight"], dev),
                gate=to_dev(x["gate"], dev), beta=to_dev(x["beta"], dev))


def _states(x, dev):
    return to_dev(x["conv_state"], dev), to_dev(x["ssm_state"], dev)


def test_noalloc_matches_the_allocating_prefill_on_two_calls():
    dev = device()
    cases = [(synth.Shape(2, 4, 64, 64, 4), [37, 100, 5, 0, 2]),   # ragged, empty and short sequences
             (synth.PRODUCTION, [256, 200])]                       # 456 tokens at D = 8192 (15.4 MB)
    for n, (shape, lengths) in enumerate(cases):
        cfg, _ = configs(shape, "bf16")
        x = synth.varlen_prefill(seed=90 + n, shape=shape, lengths=lengths)
        a = _inputs(x, dev)
        cu_host = x["cu_seqlens"]
        N, T = len(cu_host) - 1, int(cu_host[-1])
        out_shape = (T, shape.num_v_heads, shape.head_v_dim)

        conv_ref, S_ref = _states(x, dev)
        out_ref = torch.empty(out_shape, device=dev)
        ws = torch.empty(gb.gdn_prefill_workspace_size(cfg, N, T), dtype=torch.uint8, device=dev)
        gb.gdn_forward_prefill(cfg, N, a["cu"], cu_host, a["qkv"], a["w"], a["gate"], a["beta"], conv_ref, S_ref,
                               out_ref, gb.GDN_PREFILL_RESIDENT, ws)

        conv, S = _states(x, dev)
        out = torch.full(out_shape, float("nan"), device=dev)
        gb.gdn_forward_prefill_noalloc(cfg, N, a["cu"], cu_host, a["qkv"], a["w"], a["gate"], a["beta"], conv, S,
                                       out)
        torch.cuda.synchronize()
        # the same kernels on the same inputs, only the workspace address differs: bit for bit
        assert np.array_equal(bits(out), bits(out_ref)), f"call {n}: output"
        assert np.array_equal(bits(S), bits(S_ref)), f"call {n}: recurrent state"
        assert np.array_equal(bits(conv), bits(conv_ref)), f"call {n}: conv state"
        assert_parity(f64(out), f64(out_ref), f64(S), f64(S_ref), what=f"call {n}")


def test_noalloc_rejects_a_problem_larger_than_its_scratch():
    dev = device()
    cfg, _ = configs(synth.PRODUCTION, "bf16")
    T = 497                                   # 497 * (4 * 8192 + 64 * 16) bytes > 16 MiB
    cu = np.array([0, T], np.int32)
    x = torch.zeros(T * cfg.D, dtype=torch.bfloat16, device=dev)
    g = torch.zeros(T * 32, device=dev)
    w = torch.zeros(cfg.D * 4, dtype=torch.bfloat16, device=dev)
    conv = torch.zeros(cfg.D * 3, dtype=torch.bfloat16, device=dev)
    S = torch.zeros(32 * 128 * 128, device=dev)
    out = torch.zeros(T * 32 * 128, device=dev)
    with pytest.raises(gb.GdnError) as e:
        gb.gdn_forward_prefill_noalloc(cfg, 1, to_dev(cu, dev), cu, x, w, g, g, conv, S, out)
    assert e.value.status == 9
