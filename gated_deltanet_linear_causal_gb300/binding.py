"""Python binding of the C ABI in include/gdn.h (ctypes; argument marshalling only).

Every function has the name of the C entry point it calls.  Tensors are torch
tensors already on the GPU (the library computes nothing on the host); the
binding checks that each one is contiguous, on CUDA, of the right dtype and
large enough for the shape the call implies, so that a mistake becomes a Python
exception instead of an out-of-bounds access on the device.  Then it passes raw
pointers and the current torch stream to the library.

The library is built in-tree by ``gated_deltanet_linear_causal_gb300.build``;
if it is missing, loading fails loudly: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

GDN_OK = 0
GDN_ERR_RANGE = 10
GDN_BF16, GDN_F32 = 0, 1
GDN_PREFILL_RESIDENT, GDN_PREFILL_CHUNKED = 0, 1

EXPORTED = ("gdn_conv_state_init", "gdn_forward_decode", "gdn_prefill_workspace_size", "gdn_forward_prefill",
            "gdn_forward_verify", "gdn_verify_commit", "gdn_status_string", "gdn_last_cuda_error",
            "gdn_device_error", "gdn_gated_rmsnorm", "gdn_forward_decode_gated", "gdn_forward_prefill_gated")


class GdnError(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn}: status {status} ({msg})")
        self.status = status


class gdn_config_t(ctypes.Structure):
    _fields_ = [("num_k_heads", ctypes.c_int32), ("num_v_heads", ctypes.c_int32),
                ("head_k_dim", ctypes.c_int32), ("head_v_dim", ctypes.c_int32),
                ("conv_kernel", ctypes.c_int32), ("use_qk_l2norm", ctypes.c_int32),
                ("l2norm_eps", ctypes.c_float), ("io_dtype", ctypes.c_int32),
                ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p)]

    @property
    def D(self):
        return 2 * self.num_k_heads * self.head_k_dim + self.num_v_heads * self.head_v_dim

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.io_dtype == GDN_BF16 else torch.float32


def make_config(num_k_heads, num_v_heads, head_k_dim, head_v_dim, conv_kernel=4, use_qk_l2norm=True,
                l2norm_eps=1e-6, io_dtype="bf16", A_log=None, dt_bias=None) -> gdn_config_t:
    """A_log, dt_bias: optional CUDA fp32 tensors of num_v_heads; when given, the gate
    and beta tensors of every call are the raw projections a and b (see include/gdn.h).
    The config keeps references to them for as long as it lives."""
    io = {"bf16": GDN_BF16, "f32": GDN_F32}[io_dtype] if isinstance(io_dtype, str) else int(io_dtype)
    if (A_log is None) != (dt_bias is None):
        raise ValueError("A_log and dt_bias go together")
    ptrs = (None, None)
    if A_log is not None:
        for name, t in (("A_log", A_log), ("dt_bias", dt_bias)):
            if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()
                    and t.numel() == num_v_heads):
                raise ValueError(f"{name}: expected a contiguous CUDA float32 tensor of {num_v_heads} elements")
        ptrs = (A_log.data_ptr(), dt_bias.data_ptr())
    cfg = gdn_config_t(num_k_heads, num_v_heads, head_k_dim, head_v_dim, conv_kernel, int(bool(use_qk_l2norm)),
                       l2norm_eps, io, *ptrs)
    cfg._keep = (A_log, dt_bias)
    return cfg


_lib = None


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load libgdn.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        p = path or _build.LIB
        if not os.path.exists(p):
            raise RuntimeError(f"CUDA library not built: {p} (run __graft_entry__.build())")
        lib = ctypes.CDLL(p)
        vp, i32, i64, st = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        cfgp = ctypes.POINTER(gdn_config_t)
        lib.gdn_conv_state_init.argtypes = [cfgp, i32, vp, vp, vp]
        lib.gdn_forward_decode.argtypes = [cfgp, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.gdn_prefill_workspace_size.argtypes = [cfgp, i32, i64, i32]
        lib.gdn_prefill_workspace_size.restype = st
        lib.gdn_forward_prefill.argtypes = [cfgp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, st, vp]
        lib.gdn_forward_verify.argtypes = [cfgp, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.gdn_verify_commit.argtypes = [cfgp, i32, i32, vp, vp, vp, vp, vp, vp, vp]
        lib.gdn_status_string.argtypes = [i32]
        lib.gdn_status_string.restype = ctypes.c_char_p
        lib.gdn_last_cuda_error.argtypes = []
        lib.gdn_last_cuda_error.restype = i32
        lib.gdn_device_error.argtypes = [ctypes.POINTER(i32), i32]
        lib.gdn_device_error.restype = i32
        lib.gdn_gated_rmsnorm.argtypes = [cfgp, i64, vp, vp, vp, ctypes.c_float, vp, vp]
        lib.gdn_forward_decode_gated.argtypes = [cfgp, i32, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp]
        lib.gdn_forward_prefill_gated.argtypes = [cfgp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float,
                                                  vp, i32, vp, st, vp]
        for name in ("gdn_conv_state_init", "gdn_forward_decode", "gdn_forward_prefill", "gdn_forward_verify",
                     "gdn_verify_commit", "gdn_gated_rmsnorm", "gdn_forward_decode_gated", "gdn_forward_prefill_gated"):
            getattr(lib, name).restype = i32
        _lib = lib
    return _lib


def _check(fn, status):
    if status != GDN_OK:
        lib = load()
        msg = lib.gdn_status_string(status).decode()
        if status == 6:
            msg += f"; cudaError {lib.gdn_last_cuda_error()}"
        raise GdnError(fn, status, msg)


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(name, t, dtype, numel, optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if t.numel() < numel:
        raise ValueError(f"{name}: {t.numel()} elements, needs {numel}")
    return t.data_ptr() if t.numel() else None


def gdn_conv_state_init(cfg, batch, conv_state, ssm_state, stream=None):
    D, K = cfg.D, cfg.conv_kernel
    c = _dev("conv_state", conv_state, cfg.torch_dtype, batch * D * (K - 1), optional=True)
    s = _dev("ssm_state", ssm_state, torch.float32, batch * cfg.num_v_heads * cfg.head_k_dim * cfg.head_v_dim,
             optional=True)
    _check("gdn_conv_state_init", load().gdn_conv_state_init(ctypes.byref(cfg), batch, c, s, _stream(stream)))


def gdn_forward_decode(cfg, batch, qkv, conv_weight, gate, beta, conv_state, ssm_state, out, stream=None):
    if batch == 0:
        return
    D, K, H = cfg.D, cfg.conv_kernel, cfg.num_v_heads
    io = cfg.torch_dtype
    args = [_dev("qkv", qkv, io, batch * D), _dev("conv_weight", conv_weight, io, D * K),
            _dev("gate", gate, torch.float32, batch * H), _dev("beta", beta, torch.float32, batch * H),
            _dev("conv_state", conv_state, io, batch * D * (K - 1)),
            _dev("ssm_state", ssm_state, torch.float32, batch * H * cfg.head_k_dim * cfg.head_v_dim),
            _dev("out", out, torch.float32, batch * H * cfg.head_v_dim)]
    _check("gdn_forward_decode", load().gdn_forward_decode(ctypes.byref(cfg), batch, *args, _stream(stream)))


def gdn_gated_rmsnorm(cfg, rows, o, z, weight, eps, y, stream=None):
    """Gated RMSNorm (section 2) over rows of head_v_dim: y = weight * o / rms(o) * silu(z).
    o: CUDA fp32 [rows, dv]; z, y: io dtype [rows, dv]; weight: fp32 [dv]."""
    if rows == 0:
        return
    dv, io = cfg.head_v_dim, cfg.torch_dtype
    args = [_dev("o", o, torch.float32, rows * dv), _dev("z", z, io, rows * dv), _dev("weight", weight, torch.float32, dv)]
    _check("gdn_gated_rmsnorm", load().gdn_gated_rmsnorm(ctypes.byref(cfg), rows, *args, float(eps),
                                                         _dev("y", y, io, rows * dv), _stream(stream)))


def gdn_forward_decode_gated(cfg, batch, qkv, conv_weight, gate, beta, conv_state, ssm_state, z, norm_weight, norm_eps,
                             y, stream=None):
    """gdn_forward_decode with the gated RMSNorm fused into the output: y (io dtype
    [batch, Hv, dv]) instead of the fp32 output."""
    if batch == 0:
        return
    D, K, H, dv = cfg.D, cfg.conv_kernel, cfg.num_v_heads, cfg.head_v_dim
    io = cfg.torch_dtype
    args = [_dev("qkv", qkv, io, batch * D), _dev("conv_weight", conv_weight, io, D * K),
            _dev("gate", gate, torch.float32, batch * H), _dev("beta", beta, torch.float32, batch * H),
            _dev("conv_state", conv_state, io, batch * D * (K - 1)),
            _dev("ssm_state", ssm_state, torch.float32, batch * H * cfg.head_k_dim * dv),
            _dev("z", z, io, batch * H * dv), _dev("norm_weight", norm_weight, torch.float32, dv)]
    _check("gdn_forward_decode_gated", load().gdn_forward_decode_gated(ctypes.byref(cfg), batch, *args,
                                                                       float(norm_eps),
                                                                       _dev("y", y, io, batch * H * dv),
                                                                       _stream(stream)))


def gdn_prefill_workspace_size(cfg, num_seqs, total_tokens, variant=GDN_PREFILL_RESIDENT):
    return int(load().gdn_prefill_workspace_size(ctypes.byref(cfg), num_seqs, total_tokens, variant))


def gdn_forward_prefill(cfg, num_seqs, cu_seqlens, cu_seqlens_host, qkv, conv_weight, gate, beta, conv_state,
                        ssm_state, out, variant=GDN_PREFILL_RESIDENT, workspace=None, stream=None):
    """cu_seqlens: CUDA int32 [N+1]; cu_seqlens_host: CPU int32 tensor (or numpy array) with the same values."""
    host = torch.as_tensor(cu_seqlens_host, dtype=torch.int32).contiguous()
    if host.is_cuda or host.numel() < num_seqs + 1:
        raise ValueError("cu_seqlens_host: host int32 tensor of num_seqs+1 entries")
    T = int(host[num_seqs]) if num_seqs > 0 else 0
    if T == 0:
        return
    D, K, H = cfg.D, cfg.conv_kernel, cfg.num_v_heads
    io = cfg.torch_dtype
    ws_need = gdn_prefill_workspace_size(cfg, num_seqs, T, variant)
    ws_ptr = _dev("workspace", workspace, torch.uint8, ws_need, optional=ws_need == 0)
    args = [_dev("cu_seqlens", cu_seqlens, torch.int32, num_seqs + 1), host.data_ptr(),
            _dev("qkv", qkv, io, D * T), _dev("conv_weight", conv_weight, io, D * K),
            _dev("gate", gate, torch.float32, T * H), _dev("beta", beta, torch.float32, T * H),
            _dev("conv_state", conv_state, io, num_seqs * D * (K - 1)),
            _dev("ssm_state", ssm_state, torch.float32, num_seqs * H * cfg.head_k_dim * cfg.head_v_dim),
            _dev("out", out, torch.float32, T * H * cfg.head_v_dim)]
    ws_bytes = workspace.numel() if workspace is not None else 0
    _check("gdn_forward_prefill", load().gdn_forward_prefill(ctypes.byref(cfg), num_seqs, *args, variant, ws_ptr,
                                                             ws_bytes, _stream(stream)))


def gdn_forward_prefill_gated(cfg, num_seqs, cu_seqlens, cu_seqlens_host, qkv, conv_weight, gate, beta, conv_state,
                              ssm_state, z, norm_weight, norm_eps, y, variant=GDN_PREFILL_RESIDENT, workspace=None,
                              stream=None):
    """gdn_forward_prefill with the gated RMSNorm fused into the output: y (io dtype
    [T, Hv, dv]) from z (io dtype [T, Hv, dv]) instead of the fp32 output."""
    host = torch.as_tensor(cu_seqlens_host, dtype=torch.int32).contiguous()
    if host.is_cuda or host.numel() < num_seqs + 1:
        raise ValueError("cu_seqlens_host: host int32 tensor of num_seqs+1 entries")
    T = int(host[num_seqs]) if num_seqs > 0 else 0
    if T == 0:
        return
    D, K, H, dv = cfg.D, cfg.conv_kernel, cfg.num_v_heads, cfg.head_v_dim
    io = cfg.torch_dtype
    ws_need = gdn_prefill_workspace_size(cfg, num_seqs, T, variant)
    ws_ptr = _dev("workspace", workspace, torch.uint8, ws_need, optional=ws_need == 0)
    args = [_dev("cu_seqlens", cu_seqlens, torch.int32, num_seqs + 1), host.data_ptr(),
            _dev("qkv", qkv, io, D * T), _dev("conv_weight", conv_weight, io, D * K),
            _dev("gate", gate, torch.float32, T * H), _dev("beta", beta, torch.float32, T * H),
            _dev("conv_state", conv_state, io, num_seqs * D * (K - 1)),
            _dev("ssm_state", ssm_state, torch.float32, num_seqs * H * cfg.head_k_dim * dv),
            _dev("z", z, io, T * H * dv), _dev("norm_weight", norm_weight, torch.float32, dv)]
    ws_bytes = workspace.numel() if workspace is not None else 0
    _check("gdn_forward_prefill_gated",
           load().gdn_forward_prefill_gated(ctypes.byref(cfg), num_seqs, *args, float(norm_eps),
                                            _dev("y", y, io, T * H * dv), variant, ws_ptr, ws_bytes,
                                            _stream(stream)))


def gdn_forward_verify(cfg, batch, L, qkv, conv_weight, gate, beta, conv_state, ssm_state, conv_snap, ssm_snap, out,
                       stream=None):
    if batch == 0:
        return
    D, K, H = cfg.D, cfg.conv_kernel, cfg.num_v_heads
    io = cfg.torch_dtype
    S = cfg.num_v_heads * cfg.head_k_dim * cfg.head_v_dim
    args = [_dev("qkv", qkv, io, batch * D * L), _dev("conv_weight", conv_weight, io, D * K),
            _dev("gate", gate, torch.float32, batch * L * H), _dev("beta", beta, torch.float32, batch * L * H),
            _dev("conv_state", conv_state, io, batch * D * (K - 1)),
            _dev("ssm_state", ssm_state, torch.float32, batch * S),
            _dev("conv_snap", conv_snap, io, batch * L * D * (K - 1)),
            _dev("ssm_snap", ssm_snap, torch.float32, batch * L * S),
            _dev("out", out, torch.float32, batch * L * H * cfg.head_v_dim)]
    _check("gdn_forward_verify", load().gdn_forward_verify(ctypes.byref(cfg), batch, L, *args, _stream(stream)))


def gdn_verify_commit(cfg, batch, L, accepted, conv_snap, ssm_snap, conv_state, ssm_state, status=None, stream=None):
    if batch == 0:
        return
    D, K = cfg.D, cfg.conv_kernel
    io = cfg.torch_dtype
    S = cfg.num_v_heads * cfg.head_k_dim * cfg.head_v_dim
    args = [_dev("accepted", accepted, torch.int32, batch), _dev("conv_snap", conv_snap, io, batch * L * D * (K - 1)),
            _dev("ssm_snap", ssm_snap, torch.float32, batch * L * S),
            _dev("conv_state", conv_state, io, batch * D * (K - 1)),
            _dev("ssm_state", ssm_state, torch.float32, batch * S),
            _dev("status", status, torch.int32, 1, optional=True)]
    _check("gdn_verify_commit", load().gdn_verify_commit(ctypes.byref(cfg), batch, L, *args, _stream(stream)))


def gdn_status_string(status: int) -> str:
    return load().gdn_status_string(status).decode()


def gdn_last_cuda_error() -> int:
    return int(load().gdn_last_cuda_error())


def gdn_device_error(clear=False) -> int:
    """Synchronous diagnostic: the library's device-side error word (0: none)."""
    v = ctypes.c_int32(0)
    _check("gdn_device_error", load().gdn_device_error(ctypes.byref(v), int(bool(clear))))
    return int(v.value)


def gdn_forward_prefill_noalloc(cfg, num_seqs, cu_seqlens, cu_seqlens_host, qkv, conv_weight, gate, beta, conv_state,
                                ssm_state, out, stream=None):
    """Resident prefill with the library's fixed workspace (no allocation by anyone):
    for callers that cannot call cudaMalloc.  Same arguments as gdn_forward_prefill
    minus variant and workspace; its T * (4 * D + 64 * Hk)-byte workspace must fit
    GDN_NOALLOC_SCRATCH_BYTES."""
    lib = load()
    if not hasattr(lib, "_noalloc_typed"):
        vp = ctypes.c_void_p
        lib.gdn_forward_prefill_noalloc.argtypes = [ctypes.POINTER(gdn_config_t), ctypes.c_int32] + [vp] * 10
        lib.gdn_forward_prefill_noalloc.restype = ctypes.c_int32
        lib._noalloc_typed = True
    host = torch.as_tensor(cu_seqlens_host, dtype=torch.int32).contiguous()
    if host.is_cuda or host.numel() < num_seqs + 1:
        raise ValueError("cu_seqlens_host: host int32 tensor of num_seqs+1 entries")
    T = int(host[num_seqs]) if num_seqs > 0 else 0
    D, K, H = cfg.D, cfg.conv_kernel, cfg.num_v_heads
    io = cfg.torch_dtype
    args = [_dev("cu_seqlens", cu_seqlens, torch.int32, num_seqs + 1), host.data_ptr(),
            _dev("qkv", qkv, io, D * T), _dev("conv_weight", conv_weight, io, D * K),
            _dev("gate", gate, torch.float32, T * H), _dev("beta", beta, torch.float32, T * H),
            _dev("conv_state", conv_state, io, num_seqs * D * (K - 1)),
            _dev("ssm_state", ssm_state, torch.float32, num_seqs * H * cfg.head_k_dim * cfg.head_v_dim),
            _dev("out", out, torch.float32, T * H * cfg.head_v_dim)]
    _check("gdn_forward_prefill_noalloc",
           lib.gdn_forward_prefill_noalloc(ctypes.byref(cfg), num_seqs, *args, _stream(stream)))
