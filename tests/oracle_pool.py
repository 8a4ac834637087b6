"""Per-(sequence, value head) runs of the fp64 oracle in a pool of spawned processes.

Value heads are independent: head h needs only its key head's Q and K channels,
its own V channels, its gates and its state (MNN "Qwen3.5" page, section 1.2;
reverse GQA of section 1.3 maps h to key head h / f).  So the oracle of a long or
wide workload splits into one job per (sequence, head), each a one-head call of
oracle.forward_sequence on the same input bits.  The pool uses the spawn start
method: worker processes forked from a parent that has already used the GPU can
hang.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np


def _head_channels(Hk, dk, dv, f, h):
    hk = h // f
    return np.r_[hk * dk:(hk + 1) * dk, Hk * dk + hk * dk:Hk * dk + (hk + 1) * dk,
                 2 * Hk * dk + h * dv:2 * Hk * dk + (h + 1) * dv]


def _job(args):
    import oracle
    from gated_deltanet_linear_causal_gb300 import synth
    key, dims, use_l2, eps, x, w, conv, S, g, b, io = args
    dk, dv, K = dims
    sub = oracle.Cfg(1, 1, dk, dv, K, use_l2, eps)
    cvt = (lambda a: synth.as_f64(a, "bf16")) if io == "bf16" else (lambda a: np.asarray(a, np.float64))
    r = oracle.forward_sequence(sub, cvt(x), cvt(w), cvt(conv), S[None].astype(np.float64), g[:, None], b[:, None])
    return key, r["o"][:, 0], r["S"][0]


def heads_reference(ocfg, x, pairs, io="bf16", workers=None):
    """Oracle outputs and final states of the (sequence n, value head h) pairs of a packed
    prefill workload x (synth.varlen_prefill / long_prefill layout).  Returns
    {(n, h): (o [len_n, dv], S [dk, dv])}."""
    Hk, Hv, dk, dv, K = ocfg.num_k_heads, ocfg.num_v_heads, ocfg.head_k_dim, ocfg.head_v_dim, ocfg.conv_kernel
    f = Hv // Hk
    cu = x["cu_seqlens"]
    jobs = []
    for n, h in pairs:
        a, b = int(cu[n]), int(cu[n + 1])
        ch = _head_channels(Hk, dk, dv, f, h)
        jobs.append(((n, h), (dk, dv, K), ocfg.use_qk_l2norm, ocfg.l2norm_eps,
                     np.ascontiguousarray(x["qkv"][ch, a:b]), np.ascontiguousarray(x["conv_weight"][ch]),
                     np.ascontiguousarray(x["conv_state"][n][ch]), np.asarray(x["ssm_state"][n][h], np.float32),
                     np.asarray(x["gate"][a:b, h], np.float64), np.asarray(x["beta"][a:b, h], np.float64), io))
    workers = workers or max(1, min(len(jobs), os.cpu_count() or 1))
    if workers == 1:
        return {k: (o, S) for k, o, S in map(_job, jobs)}
    with mp.get_context("spawn").Pool(workers) as pool:
        return {k: (o, S) for k, o, S in pool.imap_unordered(_job, jobs)}
