"""Shared helpers of the GPU parity tests: device transfer and the parity bar.

The bar is the one stated for this layer: for bf16 (or fp32) inputs with an fp32
state, max|o_gpu - o_ref| <= 2e-3 * RMS(o_ref) and the final state's relative L2
error <= 1e-4, against the fp64 oracle on the same input bits.
"""
import numpy as np
import torch

import oracle
from gated_deltanet_linear_causal_gb300 import binding as gb
from gated_deltanet_linear_causal_gb300 import synth

O_TOL = 2e-3      # max |o_gpu - o_ref| / RMS(o_ref)
S_TOL = 1e-4      # ||S_gpu - S_ref||_2 / ||S_ref||_2


def device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    gb.load()
    return torch.device("cuda:0")


def to_dev(arr, dev):
    arr = np.ascontiguousarray(arr)
    if arr.dtype == np.uint16:
        return torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(arr).to(dev)


def f64(t):
    if isinstance(t, torch.Tensor):
        return t.detach().float().cpu().double().numpy()
    return synth.as_f64(np.asarray(t), "")


def bits(t):
    """Raw storage bits of a device tensor (bitwise comparisons)."""
    t = t.detach().contiguous().cpu()
    return t.view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.view(torch.int32).numpy()


def out_err(o_gpu, o_ref):
    o_gpu, o_ref = np.asarray(o_gpu, np.float64), np.asarray(o_ref, np.float64)
    rms = np.sqrt(np.mean(o_ref ** 2))
    return float(np.max(np.abs(o_gpu - o_ref)) / rms)


def state_err(S_gpu, S_ref):
    S_gpu, S_ref = np.asarray(S_gpu, np.float64), np.asarray(S_ref, np.float64)
    return float(np.linalg.norm(S_gpu - S_ref) / np.linalg.norm(S_ref))


def assert_parity(o_gpu, o_ref, S_gpu=None, S_ref=None, what=""):
    e = out_err(o_gpu, o_ref)
    assert e <= O_TOL, f"{what}: max|do| = {e:.3g} RMS(o) > {O_TOL}"
    if S_gpu is not None:
        s = state_err(S_gpu, S_ref)
        assert s <= S_TOL, f"{what}: state rel L2 {s:.3g} > {S_TOL}"


def configs(shape, io="bf16", use_l2=True, eps=1e-6):
    g = gb.make_config(shape.num_k_heads, shape.num_v_heads, shape.head_k_dim, shape.head_v_dim,
                       shape.conv_kernel, use_l2, eps, io)
    o = oracle.Cfg(shape.num_k_heads, shape.num_v_heads, shape.head_k_dim, shape.head_v_dim, shape.conv_kernel,
                   use_l2, eps)
    return g, o


class Guarded:
    """An output buffer with guard bands: the tensor handed to the library is the middle
    of a larger allocation whose two ends hold a NaN pattern; check() fails if a kernel
    wrote outside the buffer it was given."""

    def __init__(self, shape, dtype, dev, guard_bytes=16384):
        esize = torch.tensor([], dtype=dtype).element_size()
        self.g = guard_bytes // esize
        n = int(np.prod(shape))
        self.buf = torch.empty(n + 2 * self.g, dtype=dtype, device=dev)
        self.buf.fill_(float("nan"))
        self.t = self.buf[self.g:self.g + n].view(shape)
        self.head0 = bits(self.buf[:self.g]).copy()
        self.tail0 = bits(self.buf[self.g + n:]).copy()

    def fill_(self, value):
        self.t.fill_(value)
        return self

    def check(self, what=""):
        n = self.t.numel()
        assert np.array_equal(bits(self.buf[:self.g]), self.head0), f"{what}: write below the buffer"
        assert np.array_equal(bits(self.buf[self.g + n:]), self.tail0), f"{what}: write past the buffer"
