"""The C-ABI library: it loads, exports every entry point include/gdn.h declares,
and rejects bad arguments on the host before any launch (no GPU needed: every
call here returns from argument validation; pointers are never dereferenced)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from gated_deltanet_linear_causal_gb300 import build, binding
    build.build()
    return binding.load()


def _declared():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            names |= set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(gdn_\w+)\s*\(", txt, re.M))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"gdn_conv_state_init", "gdn_forward_decode", "gdn_forward_prefill", "gdn_forward_verify",
            "gdn_verify_commit", "gdn_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def _cfg(**kw):
    from gated_deltanet_linear_causal_gb300 import binding
    base = dict(num_k_heads=16, num_v_heads=32, head_k_dim=128, head_v_dim=128)
    base.update(kw)
    return binding.make_config(**base)


FAKE = 0x10000  # aligned, never dereferenced: every call below fails validation first


def _decode(lib, cfg, batch=1, ptrs=None):
    p = ptrs or [FAKE] * 7
    return lib.gdn_forward_decode(ctypes.byref(cfg), batch, *p, None)


def test_config_validation(lib):
    from gated_deltanet_linear_causal_gb300 import binding
    assert _decode(lib, _cfg(io_dtype=7)) == 4                 # GDN_ERR_DTYPE
    assert _decode(lib, _cfg(head_k_dim=48)) == 8              # unsupported head size
    assert _decode(lib, _cfg(head_v_dim=40)) == 8
    assert _decode(lib, _cfg(num_v_heads=24)) == 8             # Hv not a multiple of Hk
    assert _decode(lib, _cfg(conv_kernel=9)) == 8
    assert _decode(lib, _cfg(conv_kernel=0)) == 2
    assert _decode(lib, _cfg(num_k_heads=0)) == 2
    # neither decode kernel: dk=32 is outside the bulk-copy kernel, and the slice kernel's
    # cluster would need (512/32) * 4 = 64 CTAs
    assert _decode(lib, _cfg(head_k_dim=32, head_v_dim=512, num_v_heads=64)) == 8
    assert lib.gdn_forward_decode(None, 1, *[FAKE] * 7, None) == 1
    assert binding.gdn_status_string(8).startswith("shape or variant")
    # gate parameterisation: A_log and dt_bias together, 4-byte aligned
    half = _cfg()
    half.A_log = FAKE
    assert _decode(lib, half) == 1                             # dt_bias missing
    odd = _cfg()
    odd.A_log, odd.dt_bias = FAKE, FAKE + 2
    assert _decode(lib, odd) == 3
    with pytest.raises(ValueError):
        binding.make_config(16, 32, 128, 128, A_log=object())


def test_pointer_validation(lib):
    cfg = _cfg()
    assert _decode(lib, cfg, 0, [0] * 7) == 0                 # batch 0: no-op, pointers unused
    assert _decode(lib, cfg, -1) == 2
    ptrs = [FAKE] * 7
    ptrs[0] = 0
    assert _decode(lib, cfg, 1, ptrs) == 1                     # NULL qkv
    ptrs = [FAKE] * 7
    ptrs[0] = FAKE + 8
    assert _decode(lib, cfg, 1, ptrs) == 3                     # qkv not 16-byte aligned
    ptrs = [FAKE] * 7
    ptrs[5] = FAKE + 4
    assert _decode(lib, cfg, 1, ptrs) == 3                     # state not 16-byte aligned
    v = lib.gdn_forward_verify(ctypes.byref(cfg), 1, 17, *[FAKE] * 10, None)
    assert v == 2                                              # L > 16
    v = lib.gdn_verify_commit(ctypes.byref(cfg), 1, 0, *[FAKE] * 6, None)
    assert v == 2                                              # L < 1


def test_prefill_seqlens_and_workspace_validation(lib):
    from gated_deltanet_linear_causal_gb300 import binding
    cfg = _cfg()

    def call(cu, ws_bytes=1 << 40, variant=0, n=None):
        cu = np.ascontiguousarray(cu, np.int32)
        n = len(cu) - 1 if n is None else n
        return lib.gdn_forward_prefill(ctypes.byref(cfg), n, FAKE, cu.ctypes.data, *[FAKE] * 7, variant, FAKE,
                                       ws_bytes, None)

    assert call([1, 5]) == 5                                   # must start at 0
    assert call([0, 5, 3]) == 5                                # decreasing
    assert call([0, 0, 0]) == 0                                # T = 0: no-op
    assert call([0, 64], ws_bytes=16) == 9                     # workspace too small
    assert call([0, 64], variant=3) == 2
    need = binding.gdn_prefill_workspace_size(cfg, 1, 64)
    assert need == 64 * (cfg.D * 4 + cfg.num_k_heads * 64)
    assert binding.gdn_prefill_workspace_size(_cfg(io_dtype=9), 1, 64) == 0


def test_binding_rejects_cpu_tensors(lib):
    import torch
    from gated_deltanet_linear_causal_gb300 import binding
    cfg = _cfg(num_k_heads=1, num_v_heads=1, head_k_dim=32, head_v_dim=32)
    t = torch.zeros(10)
    with pytest.raises(ValueError):
        binding.gdn_forward_decode(cfg, 1, t, t, t, t, t, t, t)


def test_gated_norm_and_gated_decode_validation(lib):
    cfg = _cfg()
    F = ctypes.c_float
    # gdn_gated_rmsnorm(cfg, rows, o, z, weight, eps, y, stream)
    norm = lambda rows, p=(FAKE,) * 3, eps=1e-6, y=FAKE: lib.gdn_gated_rmsnorm(ctypes.byref(cfg), rows, *p, F(eps), y, None)
    assert norm(0) == 0                                        # no rows: no-op
    assert norm(-1) == 2
    assert norm(4, eps=-1.0) == 2                              # eps must be >= 0 and finite
    assert norm(4, eps=float("nan")) == 2
    assert norm(4, p=(0, FAKE, FAKE)) == 1                     # NULL o
    assert norm(4, p=(FAKE, FAKE + 2, FAKE)) == 3              # z not 16-byte aligned
    assert norm(4, y=FAKE + 8) == 3
    # gdn_forward_decode_gated(cfg, B, qkv, w, gate, beta, conv, S, z, norm_w, eps, y, stream)
    def dg(c, batch=1, ptrs=None, eps=1e-6, y=FAKE):
        p = ptrs or [FAKE] * 8
        return lib.gdn_forward_decode_gated(ctypes.byref(c), batch, *p[:6], p[6], p[7], F(eps), y, None)
    assert dg(_cfg(head_v_dim=64)) == 8                        # the fused norm runs in the d_v = 128 kernel only
    assert dg(cfg, batch=-1) == 2
    assert dg(cfg, eps=-1.0) == 2
    assert dg(cfg, batch=0, ptrs=[0] * 8) == 0                 # batch 0: no-op, pointers unused
    p = [FAKE] * 8
    p[6] = 0
    assert dg(cfg, ptrs=p) == 1                                # NULL z
    p = [FAKE] * 8
    p[7] = FAKE + 4
    assert dg(cfg, ptrs=p) == 3                                # norm weight not 16-byte aligned
    assert dg(cfg, y=FAKE + 2) == 3


def test_prefill_gated_validation(lib):
    cfg = _cfg()
    F = ctypes.c_float

    # gdn_forward_prefill_gated(cfg, N, cu, cu_host, qkv, w, gate, beta, conv, S, z, norm_w, eps, y,
    #                           variant, workspace, workspace_bytes, stream)
    def call(c=cfg, cu=(0, 64), eps=1e-6, z=FAKE, wgt=FAKE, y=FAKE, variant=0, ws_bytes=16, n=None):
        cu = np.ascontiguousarray(cu, np.int32)
        n = len(cu) - 1 if n is None else n
        return lib.gdn_forward_prefill_gated(ctypes.byref(c), n, FAKE, cu.ctypes.data, *[FAKE] * 6, z, wgt, F(eps), y,
                                             variant, FAKE, ws_bytes, None)

    assert call(eps=-1.0) == 2                                 # eps must be >= 0 and finite
    assert call(eps=float("inf")) == 2
    assert call(z=0) == 1 and call(wgt=0) == 1 and call(y=0) == 1
    assert call(n=0) == 0                                      # no sequences: no-op
    assert call(cu=(0, 0)) == 0                                # T = 0: no-op
    assert call(cu=(1, 64)) == 5                               # cu_seqlens must start at 0
    assert call(y=FAKE + 8) == 3                               # y, z and the weight 16-byte aligned
    assert call(z=FAKE + 4) == 3
    assert call(wgt=FAKE + 4) == 3
    # the CTAs of a value head form one cluster of at most 8: d_v <= 128 in both forms
    assert call(c=_cfg(head_v_dim=256)) == 8
    assert call(c=_cfg(head_v_dim=256), variant=1) == 8
    assert call(ws_bytes=16) == 9                              # workspace too small (checked last)
    assert call(variant=1, ws_bytes=16) == 9
