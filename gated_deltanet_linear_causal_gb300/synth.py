"""Seeded synthetic inputs for the Gated DeltaNet layer.

This module draws random numbers and rounds them to the storage types the layer
consumes; it holds none of the layer's arithmetic.  The same arrays feed the GPU
library and the fp64 CPU oracle, so both sides see identical bits.

Generator: splitmix64 over a counter (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), 53-bit uniforms, Box-Muller
normals.  Everything is numpy integer/float arithmetic, so a given seed gives the
same stream on x86-64 and aarch64 up to the last bit of libm's log/cos (which
only matters for stored fixtures; those store their inputs explicitly).

Workload recipes follow the layer description on the MNN "Qwen3.5" page (section
1.2: inputs qkv [B, D, L], gate and beta [B, L, H], conv_weight [D, 1, K]) and
the five measured configurations: oracle scale, B=64 decode, L=8192 prefill,
packed varlen prefill and MTP verify.  N(mu, sigma) takes sigma as the standard
deviation.
"""
from __future__ import annotations

import dataclasses
import numpy as np

_MASK64 = np.uint64(0xFFFFFFFFFFFFFFFF)
_GOLDEN = np.uint64(0x9E3779B97F4A7C15)


def _fnv1a64(text: str) -> int:
    h = 0xCBF29CE484222325
    for b in text.encode():
        h ^= b
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def stream_seed(seed: int, name: str) -> int:
    """Independent stream id for tensor `name` under base `seed`."""
    return (_fnv1a64(name) ^ (seed * 0xD1B54A32D192ED03)) & 0xFFFFFFFFFFFFFFFF


def splitmix64(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """n consecutive splitmix64 outputs of the stream `seed`, starting at `offset`."""
    with np.errstate(over="ignore"):
        i = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        z = np.uint64(seed) + i * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        z = z ^ (z >> np.uint64(31))
    return z


def uniform(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """Doubles in [0, 1) with 53 random bits."""
    return (splitmix64(seed, n, offset) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """Box-Muller normals: pair i uses uniforms 2i and 2i+1 of the stream."""
    m = (n + 1) // 2
    u = uniform(seed, 2 * m)
    u1 = 1.0 - u[0::2]            # (0, 1]: log is finite
    u2 = u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * m, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return mean + std * z[:n]


def randint(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    """Integers uniform in [lo, hi] inclusive (rejection-free multiply-shift, 53-bit)."""
    span = hi - lo + 1
    return lo + np.floor(uniform(seed, n) * span).astype(np.int64)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 with round-to-nearest-even; returns uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    r = (b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _softplus(x: np.ndarray) -> np.ndarray:
    return np.logaddexp(0.0, x)


def _sigmoid(x: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-x))


@dataclasses.dataclass(frozen=True)
class Shape:
    """Head configuration: the fields of MNN's LinearAttentionParam plus the conv width."""
    num_k_heads: int
    num_v_heads: int
    head_k_dim: int
    head_v_dim: int
    conv_kernel: int = 4

    @property
    def D(self) -> int:
        return 2 * self.num_k_heads * self.head_k_dim + self.num_v_heads * self.head_v_dim


ORACLE_SCALE = Shape(2, 4, 32, 32, 4)
PRODUCTION = Shape(16, 32, 128, 128, 4)


class Draw:
    """A family of named, independent streams under one base seed."""

    def __init__(self, seed: int):
        self.seed = int(seed)

    def normal(self, name, shape, mean=0.0, std=1.0):
        n = int(np.prod(shape)) if len(shape) else 1
        return normal(stream_seed(self.seed, name), n, mean, std).reshape(shape)

    def bf16(self, name, shape, mean=0.0, std=1.0):
        """uint16 bf16 bits of N(mean, std) samples (fp32 first, then RNE to bf16)."""
        return f32_to_bf16_bits(self.normal(name, shape, mean, std).astype(np.float32))

    def f32(self, name, shape, mean=0.0, std=1.0):
        return self.normal(name, shape, mean, std).astype(np.float32)

    def gate(self, name, shape, mean=0.0):
        """gate = -softplus(N(mean, 1)) as float32 (always <= 0)."""
        return (-_softplus(self.normal(name, shape, mean, 1.0))).astype(np.float32)

    def beta(self, name, shape):
        """beta = sigmoid(N(0, 1)) as float32, in (0, 1)."""
        return _sigmoid(self.normal(name, shape)).astype(np.float32)

    def ints(self, name, n, lo, hi):
        return randint(stream_seed(self.seed, name), n, lo, hi)


# ---------------------------------------------------------------------------
# Workload recipes.  Each returns a dict of host numpy arrays; bf16 tensors are
# uint16 bit arrays and carry io="bf16".
# ---------------------------------------------------------------------------

def oracle_scale(seed=1, L=64, batch=1, shape=ORACLE_SCALE, io="f32"):
    """B=1, L=64, H_k=2, H_v=4, d=32, K=4; fp32 qkv~N(0,1) [B,D,L]; w~N(0,0.5);
    gate=-softplus(N(0,1)); beta=sigmoid(N(0,1)); zero initial states."""
    d = Draw(seed)
    D, K, H = shape.D, shape.conv_kernel, shape.num_v_heads
    mk = d.f32 if io == "f32" else d.bf16
    return dict(
        shape=shape, io=io,
        qkv=mk("qkv", (batch, D, L)),
        conv_weight=mk("w", (D, K), 0.0, 0.5),
        gate=d.gate("g", (batch, L, H)),
        beta=d.beta("b", (batch, L, H)),
        conv_state=np.zeros((batch, D, K - 1), np.float32 if io == "f32" else np.uint16),
        ssm_state=np.zeros((batch, H, shape.head_k_dim, shape.head_v_dim), np.float32),
    )


def decode_state(seed=2, batch=64, shape=PRODUCTION):
    """Carried states and weights of the B=64 decode workload: fp32 S~N(0,0.02),
    bf16 conv state N(0,1) [B,D,K-1], bf16 conv weight N(0,0.5) [D,K]."""
    d = Draw(seed)
    D, K, H = shape.D, shape.conv_kernel, shape.num_v_heads
    return dict(
        shape=shape, io="bf16",
        conv_weight=d.bf16("w", (D, K), 0.0, 0.5),
        conv_state=d.bf16("conv_state", (batch, D, K - 1)),
        ssm_state=d.f32("S", (batch, H, shape.head_k_dim, shape.head_v_dim), 0.0, 0.02),
    )


def decode_step(seed=2, step=0, batch=64, shape=PRODUCTION):
    """Fresh per-step decode inputs: bf16 qkv~N(0,1) [B,D]; gate=-softplus(N(0,1)),
    beta=sigmoid(N(0,1)) [B,H_v] fp32."""
    d = Draw(seed * 1_000_003 + 7919 * (step + 1))
    H = shape.num_v_heads
    return dict(
        qkv=d.bf16("qkv", (batch, shape.D)),
        gate=d.gate("g", (batch, H)),
        beta=d.beta("b", (batch, H)),
    )


def long_prefill(seed=3, L=8192, shape=PRODUCTION):
    """B=1, L=8192: bf16 qkv~N(0,1) [1,D,L]; slow decay gate=-softplus(N(-2,1));
    beta=sigmoid(N(0,1)); bf16 conv weight N(0,0.5); zero initial states."""
    d = Draw(seed)
    D, K, H = shape.D, shape.conv_kernel, shape.num_v_heads
    return dict(
        shape=shape, io="bf16",
        cu_seqlens=np.array([0, L], np.int32),
        qkv=d.bf16("qkv", (D, L)),
        conv_weight=d.bf16("w", (D, K), 0.0, 0.5),
        gate=d.gate("g", (L, H), mean=-2.0),
        beta=d.beta("b", (L, H)),
        conv_state=np.zeros((1, D, K - 1), np.uint16),
        ssm_state=np.zeros((1, H, shape.head_k_dim, shape.head_v_dim), np.float32),
    )


def varlen_lengths(seed=4, num_seqs=16, lo=256, hi=2048):
    return Draw(seed).ints("lengths", num_seqs, lo, hi).astype(np.int32)


def varlen_prefill(seed=4, num_seqs=16, lo=256, hi=2048, shape=PRODUCTION, lengths=None):
    """Sequences with lengths U{lo..hi} packed by cu_seqlens: bf16 qkv~N(0,1) [D,T];
    gate=-softplus(N(0,1)); beta=sigmoid(N(0,1)); per-sequence random
    S~N(0,0.02) and bf16 conv state N(0,1)."""
    d = Draw(seed)
    if lengths is None:
        lengths = varlen_lengths(seed, num_seqs, lo, hi)
    lengths = np.asarray(lengths, np.int32)
    N = len(lengths)
    cu = np.zeros(N + 1, np.int32)
    cu[1:] = np.cumsum(lengths)
    T = int(cu[-1])
    D, K, H = shape.D, shape.conv_kernel, shape.num_v_heads
    return dict(
        shape=shape, io="bf16", cu_seqlens=cu,
        qkv=d.bf16("qkv", (D, T)),
        conv_weight=d.bf16("w", (D, K), 0.0, 0.5),
        gate=d.gate("g", (T, H)),
        beta=d.beta("b", (T, H)),
        conv_state=d.bf16("conv_state", (N, D, K - 1)),
        ssm_state=d.f32("S", (N, H, shape.head_k_dim, shape.head_v_dim), 0.0, 0.02),
    )


def verify_block(seed=5, batch=32, L=4, shape=PRODUCTION):
    """MTP verify: B=32 sequences, L=4 tokens each: bf16 qkv~N(0,1) [B,D,L];
    gate=-softplus(N(0,1)); beta=sigmoid(N(0,1)); random prior fp32 S~N(0,0.02)
    and bf16 conv state; accepted lengths uniform in [0, L]."""
    d = Draw(seed)
    D, K, H = shape.D, shape.conv_kernel, shape.num_v_heads
    return dict(
        shape=shape, io="bf16",
        qkv=d.bf16("qkv", (batch, D, L)),
        conv_weight=d.bf16("w", (D, K), 0.0, 0.5),
        gate=d.gate("g", (batch, L, H)),
        beta=d.beta("b", (batch, L, H)),
        conv_state=d.bf16("conv_state", (batch, D, K - 1)),
        ssm_state=d.f32("S", (batch, H, shape.head_k_dim, shape.head_v_dim), 0.0, 0.02),
        accepted=d.ints("accepted", batch, 0, L).astype(np.int32),
    )


def raw_gates(seed, lead, num_v_heads):
    """Stand-ins for the raw gate inputs of section 1.2's parameterisation (no trained
    weights exist here): projections a, b ~ N(0, 1) float32 shaped lead + (H_v,), and
    per-head A_log, dt_bias ~ N(0, 0.5) float32 [H_v]."""
    d = Draw(seed)
    shape = tuple(lead) + (num_v_heads,)
    return dict(a=d.f32("a", shape), b=d.f32("bproj", shape),
                A_log=d.f32("A_log", (num_v_heads,), 0.0, 0.5), dt_bias=d.f32("dt_bias", (num_v_heads,), 0.0, 0.5))


def as_f64(arr: np.ndarray, io: str) -> np.ndarray:
    """Exact float64 values of stored inputs (bf16 bits or float32)."""
    if arr.dtype == np.uint16:
        return bf16_bits_to_f32(arr).astype(np.float64)
    return np.asarray(arr, dtype=np.float64)
