"""Host-side checks of the seeded input generator (no GPU)."""
import numpy as np
import torch

from gated_deltanet_linear_causal_gb300 import synth


def test_bf16_rounding_matches_torch():
    x = synth.Draw(9).f32("x", (200000,), 0.0, 3.0)
    x[:4] = [0.0, -0.0, 1e-40, 3.0e38]
    ours = synth.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = synth.bf16_bits_to_f32(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_streams_are_deterministic_and_distinct():
    a = synth.Draw(1).normal("a", (1000,))
    assert np.array_equal(a, synth.Draw(1).normal("a", (1000,)))
    assert not np.allclose(a, synth.Draw(1).normal("b", (1000,)))
    assert not np.allclose(a, synth.Draw(2).normal("a", (1000,)))


def test_normal_moments():
    z = synth.normal(12345, 400000, 0.5, 2.0)
    assert abs(z.mean() - 0.5) < 0.02 and abs(z.std() - 2.0) < 0.02


def test_gate_beta_ranges():
    d = synth.Draw(3)
    g = d.gate("g", (10000,), mean=-2.0)
    b = d.beta("b", (10000,))
    assert (g <= 0).all() and (b > 0).all() and (b < 1).all()


def test_varlen_lengths_in_range():
    L = synth.varlen_lengths(4, 16, 256, 2048)
    assert L.min() >= 256 and L.max() <= 2048 and len(L) == 16
    cu = synth.varlen_prefill(4, shape=synth.Shape(1, 1, 32, 32), lengths=[3, 5])["cu_seqlens"]
    assert list(cu) == [0, 3, 8]
