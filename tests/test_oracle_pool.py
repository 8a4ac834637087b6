"""The per-(sequence, head) oracle jobs used by the full-size GPU tests reproduce the
whole-layer oracle: splitting by value head (each head with its key head's Q/K channels
and its own V channels) changes nothing, bit for bit, in a spawned pool or in process."""
import numpy as np

import oracle
from gated_deltanet_linear_causal_gb300 import synth
from oracle_pool import heads_reference


def test_heads_reference_equals_whole_layer(oracle_mod):
    shape = synth.Shape(2, 4, 32, 16, 4)
    x = synth.varlen_prefill(seed=7, shape=shape, lengths=[19, 0, 40])
    ocfg = oracle.Cfg(2, 4, 32, 16, 4, True, 1e-6)
    o, conv, S = oracle.prefill(ocfg, x["cu_seqlens"], synth.as_f64(x["qkv"], "bf16"),
                                synth.as_f64(x["conv_weight"], "bf16"), x["gate"], x["beta"],
                                synth.as_f64(x["conv_state"], "bf16"), x["ssm_state"])
    pairs = [(n, h) for n in (0, 2) for h in range(4)]
    cu = x["cu_seqlens"]
    for workers in (1, 2):
        ref = heads_reference(ocfg, x, pairs, workers=workers)
        for (n, h), (o_h, S_h) in ref.items():
            assert np.array_equal(o_h, o[cu[n]:cu[n + 1], h])
            assert np.array_equal(S_h, S[n, h])
