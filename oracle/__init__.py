"""fp64 CPU oracle for the Gated DeltaNet linear-attention layer.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The GPU library
never calls it and shares no code with it.

The arithmetic lives in ``gdn_oracle.c`` (plain C, double precision,
single-threaded, compiled with ``-ffp-contract=off``); this module compiles it
with gcc on first use and marshals numpy float64 arrays in and out.  It follows
the MNN discussion "MNN Model Support: Qwen3.5": section 1.2 (the five steps),
section 1.3 (reverse GQA) and section 1.4 (the carried conv and recurrent
states).

Layouts of the wrappers below match the GPU library's entry points:
  decode   qkv [B, D]      gate/beta [B, H_v]     out [B, H_v, d_v]
  prefill  qkv [D, T]      gate/beta [T, H_v]     out [T, H_v, d_v]   (cu_seqlens packed)
  verify   qkv [B, D, L]   gate/beta [B, L, H_v]  out [B, L, H_v, d_v]
Conv state [.., D, K-1] (oldest first); SSM state [.., H_v, d_k, d_v].
Every pinned function: see tests/test_oracle_pins.py.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdn_oracle.so")
_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]
_lock = threading.Lock()
_lib = None


def compile_source(src_path: str, out_path: str) -> str:
    """Compile one C source of the oracle into a shared library (gcc)."""
    tmp = out_path + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", *_CFLAGS, src_path, "-o", tmp, "-lm"])
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile the C oracle into oracle/_build/libgdn_oracle.so."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        compile_source(_SRC, _LIB_PATH)
    return _LIB_PATH


def open_library(path: str):
    """ctypes handle of a compiled oracle library with its signatures declared."""
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(ctypes.c_double)
    i64 = ctypes.c_int64
    lib.gdn_oracle_conv1d_silu.argtypes = [i64, i64, i64, P, P, P, P, P, P]
    lib.gdn_oracle_split_norm_scale.argtypes = [i64, i64, i64, i64, i64, ctypes.c_int,
                                                ctypes.c_double, P, P, P, P]
    lib.gdn_oracle_delta_rule.argtypes = [i64, i64, i64, i64, P, P, P, P, P, P, P, P, P, P]
    lib.gdn_oracle_forward.argtypes = [i64, i64, i64, i64, i64, ctypes.c_int, ctypes.c_double,
                                       i64, P, P, P, P, P, P, P, P, P, P, P, P]
    lib.gdn_oracle_forward_work_doubles.argtypes = [i64] * 5
    lib.gdn_oracle_forward_work_doubles.restype = i64
    lib.gdn_oracle_gate_beta.argtypes = [i64, i64, P, P, P, P, P, P]
    lib.gdn_oracle_gated_rmsnorm.argtypes = [i64, i64, P, P, P, ctypes.c_double, P]
    for f in (lib.gdn_oracle_conv1d_silu, lib.gdn_oracle_split_norm_scale,
              lib.gdn_oracle_delta_rule, lib.gdn_oracle_forward, lib.gdn_oracle_gate_beta,
              lib.gdn_oracle_gated_rmsnorm):
        f.restype = None
    return lib


class use_library:
    """Context manager: run the wrappers of this module on another compiled oracle
    library (the mutation tests load deliberately broken copies this way)."""

    def __init__(self, path: str):
        self.lib = open_library(path)

    def __enter__(self):
        global _lib
        _lock.acquire()
        self.prev, _lib = _lib, self.lib
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.prev
        _lock.release()
        return False


def _load():
    global _lib
    if _lib is None:
        _lib = open_library(build())
    return _lib


def _in(a, shape=None):
    a = np.ascontiguousarray(a, dtype=np.float64)
    if shape is not None:
        assert a.shape == tuple(shape), (a.shape, shape)
    return a


def _p(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


@dataclasses.dataclass(frozen=True)
class Cfg:
    """LinearAttentionParam of the MNN page (section 1.4) plus conv width and eps."""
    num_k_heads: int
    num_v_heads: int
    head_k_dim: int
    head_v_dim: int
    conv_kernel: int = 4
    use_qk_l2norm: bool = True
    l2norm_eps: float = 1e-6

    @property
    def D(self):
        return 2 * self.num_k_heads * self.head_k_dim + self.num_v_heads * self.head_v_dim


# ---------------------------------------------------------------------------
# Single steps (each pinned on its own by the tests).
# ---------------------------------------------------------------------------

def gate_beta(a, b, A_log, dt_bias):
    """Gate parameterisation of section 1.2: from the raw projections a, b [.., H]
    and the per-head A_log, dt_bias [H], gate = -exp(A_log) * softplus(a + dt_bias)
    and beta = sigmoid(b).  Returns (gate, beta), float64, shaped like a."""
    a = _in(a)
    b = _in(b, a.shape)
    H = a.shape[-1]
    A_log = _in(A_log, (H,))
    dt_bias = _in(dt_bias, (H,))
    gate, beta = np.empty_like(a), np.empty_like(a)
    _load().gdn_oracle_gate_beta(a.size // H, H, _p(a), _p(b), _p(A_log), _p(dt_bias), _p(gate), _p(beta))
    return gate, beta


def gated_rmsnorm(o, z, weight, eps):
    """Gated RMSNorm of section 2 over the last axis: weight * o / sqrt(mean(o^2) + eps)
    * silu(z).  o, z [.., n]; weight [n].  Returns float64 shaped like o."""
    o = _in(o)
    z = _in(z, o.shape)
    n = o.shape[-1]
    weight = _in(weight, (n,))
    y = np.empty_like(o)
    _load().gdn_oracle_gated_rmsnorm(o.size // n, n, _p(o), _p(z), _p(weight), float(eps), _p(y))
    return y


def conv1d_silu(x, w, state_in, snapshots=False):
    """Step 1 over one sequence. x [D, L], w [D, K], state_in [D, K-1].
    Returns (y [D, L], state_out [D, K-1], conv_snap [L, D, K-1] or None)."""
    x = _in(x)
    D, L = x.shape
    w = _in(w)
    K = w.shape[1]
    state_in = _in(state_in, (D, K - 1))
    y = np.empty((D, L))
    st = np.empty((D, K - 1))
    snap = np.empty((L, D, K - 1)) if snapshots else None
    _load().gdn_oracle_conv1d_silu(D, K, L, _p(x), _p(w), _p(state_in), _p(y), _p(st), _p(snap))
    return y, st, snap


def split_norm_scale(cfg: Cfg, y):
    """Steps 2-4 over one sequence's conv output y [D, L].
    Returns q, k [L, H_v, d_k] (GQA-expanded) and v [L, H_v, d_v]."""
    y = _in(y)
    D, L = y.shape
    assert D == cfg.D
    H, dk, dv = cfg.num_v_heads, cfg.head_k_dim, cfg.head_v_dim
    q = np.empty((L, H, dk)); k = np.empty((L, H, dk)); v = np.empty((L, H, dv))
    _load().gdn_oracle_split_norm_scale(cfg.num_k_heads, H, dk, dv, L, int(cfg.use_qk_l2norm),
                                        float(cfg.l2norm_eps), _p(y), _p(q), _p(k), _p(v))
    return q, k, v


def delta_rule(q, k, v, g, beta, S0, snapshots=False):
    """Step 5. q, k [L, H, d_k]; v [L, H, d_v]; g, beta [L, H]; S0 [H, d_k, d_v].
    Returns (o [L, H, d_v], S [H, d_k, d_v], S_snap [L, H, d_k, d_v] or None)."""
    q = _in(q); k = _in(k); v = _in(v)
    L, H, dk = q.shape
    dv = v.shape[2]
    g = _in(g, (L, H)); beta = _in(beta, (L, H)); S0 = _in(S0, (H, dk, dv))
    o = np.empty((L, H, dv)); S = np.empty((H, dk, dv))
    snap = np.empty((L, H, dk, dv)) if snapshots else None
    work = np.empty(dk * dv + 2 * dv)
    _load().gdn_oracle_delta_rule(H, dk, dv, L, _p(q), _p(k), _p(v), _p(g), _p(beta), _p(S0),
                                  _p(o), _p(S), _p(snap), _p(work))
    return o, S, snap


def forward_sequence(cfg: Cfg, x, w, conv_in, S_in, g, beta, snapshots=False):
    """All five steps over one sequence.  x [D, L]; w [D, K]; conv_in [D, K-1];
    S_in [H_v, d_k, d_v]; g, beta [L, H_v].  Returns dict o [L, H_v, d_v],
    conv [D, K-1], S [H_v, d_k, d_v] and, with snapshots, conv_snap [L, D, K-1],
    S_snap [L, H_v, d_k, d_v]."""
    D, K, H = cfg.D, cfg.conv_kernel, cfg.num_v_heads
    dk, dv = cfg.head_k_dim, cfg.head_v_dim
    x = _in(x)
    L = x.shape[1]
    assert x.shape[0] == D
    w = _in(w, (D, K)); conv_in = _in(conv_in, (D, K - 1)); S_in = _in(S_in, (H, dk, dv))
    g = _in(g, (L, H)); beta = _in(beta, (L, H))
    lib = _load()
    work = np.empty(max(1, lib.gdn_oracle_forward_work_doubles(cfg.num_k_heads, H, dk, dv, L)))
    o = np.empty((L, H, dv)); conv = np.empty((D, K - 1)); S = np.empty((H, dk, dv))
    cs = np.empty((L, D, K - 1)) if snapshots else None
    ss = np.empty((L, H, dk, dv)) if snapshots else None
    lib.gdn_oracle_forward(cfg.num_k_heads, H, dk, dv, K, int(cfg.use_qk_l2norm), float(cfg.l2norm_eps),
                           L, _p(x), _p(w), _p(conv_in), _p(S_in), _p(g), _p(beta), _p(o), _p(conv),
                           _p(S), _p(cs), _p(ss), _p(work))
    out = dict(o=o, conv=conv, S=S)
    if snapshots:
        out.update(conv_snap=cs, S_snap=ss)
    return out


# ---------------------------------------------------------------------------
# Entry-point-shaped wrappers: one sequence at a time, in plain loops.
# ---------------------------------------------------------------------------

def decode(cfg: Cfg, qkv, w, gate, beta, conv_state, ssm_state, batch_index=None):
    """One decode step (L=1) for each sequence b in `batch_index` (all by default).
    qkv [B, D]; gate, beta [B, H_v]; conv_state [B, D, K-1]; ssm_state [B, H_v, d_k, d_v].
    Returns out [n, H_v, d_v], conv [n, D, K-1], S [n, H_v, d_k, d_v] for those sequences."""
    B = qkv.shape[0]
    idx = range(B) if batch_index is None else batch_index
    outs, convs, Ss = [], [], []
    for b in idx:
        r = forward_sequence(cfg, np.asarray(qkv[b], np.float64)[:, None], w, conv_state[b], ssm_state[b],
                             np.asarray(gate[b])[None, :], np.asarray(beta[b])[None, :])
        outs.append(r["o"][0]); convs.append(r["conv"]); Ss.append(r["S"])
    return np.stack(outs), np.stack(convs), np.stack(Ss)


def prefill(cfg: Cfg, cu_seqlens, qkv, w, gate, beta, conv_state, ssm_state, seq_index=None):
    """Packed varlen prefill: sequence n covers tokens [cu[n], cu[n+1]) of qkv [D, T],
    gate/beta [T, H_v]; each starts from its own conv_state[n], ssm_state[n] and
    the conv window never crosses a sequence boundary.
    Returns out [T, H_v, d_v] (rows of unselected sequences are NaN), conv [N, D, K-1],
    S [N, H_v, d_k, d_v] (unselected sequences keep their input state)."""
    cu = np.asarray(cu_seqlens, np.int64)
    N = len(cu) - 1
    T = int(cu[-1])
    out = np.full((T, cfg.num_v_heads, cfg.head_v_dim), np.nan)
    conv = np.array(conv_state, np.float64, copy=True)
    S = np.array(ssm_state, np.float64, copy=True)
    for n in (range(N) if seq_index is None else seq_index):
        a, b = int(cu[n]), int(cu[n + 1])
        r = forward_sequence(cfg, np.asarray(qkv[:, a:b], np.float64), w, conv_state[n], ssm_state[n],
                             gate[a:b], beta[a:b])
        out[a:b] = r["o"]; conv[n] = r["conv"]; S[n] = r["S"]
    return out, conv, S


def verify(cfg: Cfg, qkv, w, gate, beta, conv_state, ssm_state, batch_index=None):
    """MTP verify: sequence b runs its L draft tokens qkv[b] [D, L] from the prior states.
    Returns out [n, L, H_v, d_v], conv_snap [n, L, D, K-1], S_snap [n, L, H_v, d_k, d_v];
    snapshot t is the state after tokens 0..t."""
    B = qkv.shape[0]
    idx = range(B) if batch_index is None else batch_index
    o, cs, ss = [], [], []
    for b in idx:
        r = forward_sequence(cfg, qkv[b], w, conv_state[b], ssm_state[b], gate[b], beta[b], snapshots=True)
        o.append(r["o"]); cs.append(r["conv_snap"]); ss.append(r["S_snap"])
    return np.stack(o), np.stack(cs), np.stack(ss)


def commit(conv_state, ssm_state, conv_snap, ssm_snap, accepted):
    """Roll back to the accepted prefix: sequence b takes snapshot accepted[b]-1,
    or keeps its prior state when accepted[b] == 0."""
    conv = np.array(conv_state, np.float64, copy=True)
    S = np.array(ssm_state, np.float64, copy=True)
    for b, a in enumerate(np.asarray(accepted)):
        if a > 0:
            conv[b] = conv_snap[b, a - 1]
            S[b] = ssm_snap[b, a - 1]
    return conv, S
