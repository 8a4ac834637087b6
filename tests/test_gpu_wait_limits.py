"""The bounded waits behind every kernel's failure detection, exercised on the GPU.

Every device-side wait in the library (mbarrier phases of bulk copies and MMAs, the
cluster exchange of the fused norms) gives up after 2 s of the global timer and reports
failure: the kernel sets the device error word (`gdn_device_error`), lets its own
copies land and returns, instead of hanging or trapping.  These tests drive the same
helpers (`gdn_tma.cuh`) from a test-only kernel: a wait on a phase that nothing
completes must give up after about 2 s, a wait that watches an abort flag must
return once another warp sets it, a completed phase must return at once, and the
context must stay usable afterwards (a decode call still matches the oracle).
"""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_linear_causal_gb300 import binding as gb
from gated_deltanet_linear_causal_gb300 import synth
from gdn_testutil import assert_parity, configs, device, f64, to_dev

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "gated_deltanet_linear_causal_gb300", "csrc")


@pytest.fixture(scope="module")
def waitlib():
    device()
    nvcc = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
    tmp = tempfile.mkdtemp(prefix="gdn_wait_")
    so = os.path.join(tmp, "libwaittest.so")
    subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-Xcompiler",
                           "-fPIC", "-shared", "-I", CSRC, os.path.join(HERE, "csrc", "wait_limits.cu"), "-o", so,
                           "-lcudart"])
    lib = ctypes.CDLL(so)
    lib.gdn_test_wait.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_longlong)]
    lib.gdn_test_wait.restype = ctypes.c_int
    return lib


def _run(lib, mode):
    out = (ctypes.c_longlong * 2)()
    rc = lib.gdn_test_wait(mode, out)
    assert rc == 0, f"CUDA error {rc}"
    return int(out[0]), int(out[1]) * 1e-9


def test_wait_on_a_phase_nothing_completes_gives_up(waitlib):
    ok, secs = _run(waitlib, 0)
    assert ok == 0, "a wait on a phase that never completes reported success"
    assert 1.9 <= secs < 5.0, f"the bounded wait took {secs:.2f} s"
    print(f"bounded wait gave up after {secs:.3f} s")


def test_wait_returns_when_abort_is_set(waitlib):
    ok, secs = _run(waitlib, 1)
    assert ok == 0
    assert secs < 0.1, f"the abort flag took {secs:.4f} s to end the wait"


def test_completed_phase_returns_at_once(waitlib):
    ok, secs = _run(waitlib, 2)
    assert ok == 1
    assert secs < 0.01


def test_context_usable_after_timeouts(waitlib):
    for mode in (0, 1):
        _run(waitlib, mode)
    dev = device()
    shape = synth.Shape(2, 4, 128, 128, 4)
    cfg, ocfg = configs(shape, "bf16")
    B = 3
    st = synth.decode_state(71, B, shape)
    d = synth.decode_step(71, 0, B, shape)
    conv, S = to_dev(st["conv_state"], dev), to_dev(st["ssm_state"], dev)
    out = torch.empty(B, shape.num_v_heads, shape.head_v_dim, device=dev)
    gb.gdn_forward_decode(cfg, B, to_dev(d["qkv"], dev), to_dev(st["conv_weight"], dev), to_dev(d["gate"], dev),
                          to_dev(d["beta"], dev), conv, S, out)
    o_r, _, S_r = oracle.decode(ocfg, f64(d["qkv"]), f64(st["conv_weight"]), d["gate"], d["beta"],
                                f64(st["conv_state"]), st["ssm_state"].astype(np.float64))
    torch.cuda.synchronize()
    assert_parity(f64(out), o_r, f64(S), S_r, what="decode after the timeouts")
    assert gb.gdn_device_error() == 0
