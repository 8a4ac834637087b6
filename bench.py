#!/usr/bin/env python3
"""Throughput of the Gated DeltaNet layer on GB300: one JSON line on stdout.

Headline ("step" = one decode call over a batch of 64 sequences, every step of
the layer in one kernel): B=64, H_k=16, H_v=32, d_k=d_v=128, K=4, bf16 qkv,
carried fp32 state, fresh seeded inputs each step.  Two state sets rotate so
that each step reads its state from HBM (2 x 134 MB > the 126 MB L2).

Also reported on the same line (N=1 only): the L=8192 prefill, the packed
varlen prefill (16 sequences, lengths U{256..2048}) and the B=32, L=4 MTP
verify + commit.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle on the host cores instead (the
page describes no GPU implementation to compare with).  Under torchrun, ranks
run independent replicas (the layer has no cross-sequence exchange): rank 0
prints, value = tokens of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN layer tokens/s (decode B=64, prefill L=8192); % of GB300 HBM roofline"
B_DECODE, N_INPUT_STEPS = 64, 256


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


_CODE_TOKENS = re.compile(r'"(?:\\.|[^"\\])*"|/\*.*?\*/|//[^\n]*|\s+', re.S)


def _code_only(text):
    """Source text with comments removed and every run of whitespace made one space (string
    literals otherwise kept), so that an edit to comments or layout does not count as a change
    of the kernel."""
    def keep(m):
        t = m.group(0)
        return t if t.startswith('"') else " "
    return re.sub(r"\s+", " ", _CODE_TOKENS.sub(keep, text)).strip()


def _source_sha(names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "gated_deltanet_linear_causal_gb300", "csrc", n), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def _traffic(kernel_key, sources, profile="stream_kernel_decode_b64.json", field="dram_bytes_per_launch"):
    """DRAM bytes per launch (or per call) from a committed ncu summary, or None if the
    kernels' sources changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", profile)
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel_key)
    if not d or d.get("source_sha") != _source_sha(sources):
        return None
    return d.get(field)


class ClockSampler:
    """nvidia-smi clock/throttle sampling while the GPU is under the bench's load."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.proc = index, None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        return dist, dist.get_rank(), ws
    return None, 0, 1


def _max_over_ranks(dist, ms, dev):
    """The job's time: the slowest rank's (every rank passes its own)."""
    if not dist:
        return ms
    import torch
    t = torch.tensor([ms], device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_value(units_per_rank, world, ms):
    """Whole-job throughput: the units all ranks processed over the job's time."""
    return units_per_rank * world / (ms / 1e3)


def _to_dev(arr, dev):
    import numpy as np
    import torch
    arr = np.ascontiguousarray(arr)
    if arr.dtype == np.uint16:
        return torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(arr).to(dev)


def _pinned(arr):
    import numpy as np
    import torch
    arr = np.ascontiguousarray(arr)
    t = torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16) if arr.dtype == np.uint16 else torch.from_numpy(arr)
    return t.pin_memory()


# ---------------------------------------------------------------------------
# Workloads on the GPU
# ---------------------------------------------------------------------------

def decode_bytes(shape, B):
    """Algorithmic HBM bytes of one decode call: S read+write, qkv, conv state read+write,
    output, conv weight, gate and beta."""
    S = B * shape.num_v_heads * shape.head_k_dim * shape.head_v_dim * 4
    return (2 * S + B * shape.D * 2 + 2 * B * shape.D * (shape.conv_kernel - 1) * 2 +
            B * shape.num_v_heads * shape.head_v_dim * 4 + shape.D * shape.conv_kernel * 2 +
            2 * B * shape.num_v_heads * 4)


def prefill_bytes(shape, cu, random_state):
    """qkv in, fp32 output, gate and beta, conv weight, states (final write; plus the
    initial read when the sequences start from a given state)."""
    import numpy as np
    T, N = int(cu[-1]), len(cu) - 1
    S = N * shape.num_v_heads * shape.head_k_dim * shape.head_v_dim * 4
    conv = N * shape.D * (shape.conv_kernel - 1) * 2
    return (T * shape.D * 2 + T * shape.num_v_heads * shape.head_v_dim * 4 + 2 * T * shape.num_v_heads * 4 +
            shape.D * shape.conv_kernel * 2 + (2 if random_state else 1) * (S + conv))


def chunked_tensor_flops(shape, cu, C=64):
    """Tensor-core flops of one chunked prefill call (64-token chunks), as the products are
    defined (algorithmic) and as issued (every product takes fp32 operands as bf16 hi/lo
    pairs: three bf16 products each).  Per (chunk, key head): [K; Q] K^T; per (chunk,
    value head): W = T diag(beta gamma) K and u = T diag(beta) V, then the chain's
    [W; Q~] S0, K~^T U and [P; P] U (P stacked twice so that it accumulates onto the
    Q~ S0 rows)."""
    dk, dv, f = shape.head_k_dim, shape.head_v_dim, shape.num_v_heads // shape.num_k_heads
    nchunk = sum((int(cu[i + 1]) - int(cu[i]) + C - 1) // C for i in range(len(cu) - 1))
    gram = 2 * (2 * C) * C * dk
    per_vhead = 2 * C * dk * C + 2 * C * dv * C + 2 * (2 * C) * dv * dk + 2 * dk * dv * C + 2 * (2 * C) * dv * C
    per_pair = gram + f * per_vhead
    issued = 3 * per_pair * nchunk * shape.num_k_heads
    return issued // 3, issued


def prefill_roofline(nbytes, flops_issued, ms, peaks):
    """The larger of the HBM bound (algorithmic bytes / measured copy bandwidth) and the
    tensor bound (issued flops / measured sustained bf16 rate) against the measured time."""
    hbm_us = nbytes / (peaks["hbm_gbs"] * 1e9) * 1e6
    tensor_us = flops_issued / (peaks["bf16_tflops_sustained"] * 1e12) * 1e6
    bound_us = max(hbm_us, tensor_us)
    return {"hbm_bound_us": round(hbm_us, 2), "tensor_bound_us": round(tensor_us, 2),
            "bound": "hbm" if hbm_us >= tensor_us else "tensor", "bound_us": round(bound_us, 2),
            "frac": round(bound_us / (ms * 1e3), 4)}


def verify_bytes(shape, B, L):
    S = B * shape.num_v_heads * shape.head_k_dim * shape.head_v_dim * 4
    conv = B * shape.D * (shape.conv_kernel - 1) * 2
    return (S + L * S + conv + L * conv + B * L * shape.D * 2 + B * L * shape.num_v_heads * shape.head_v_dim * 4 +
            2 * B * L * shape.num_v_heads * 4 + shape.D * shape.conv_kernel * 2)


def decode_inputs(args, rank):
    from gated_deltanet_linear_causal_gb300 import synth
    shape = synth.PRODUCTION
    st = synth.decode_state(2 + 1000 * rank, B_DECODE, shape)
    n_in = min(N_INPUT_STEPS, max(args.steps, 1) + args.warmup)
    steps = [synth.decode_step(2 + 1000 * rank, s, B_DECODE, shape) for s in range(n_in)]
    return st, steps


def run_decode(args, dev, dist, rank, world, st, steps):
    import numpy as np
    import torch
    from gated_deltanet_linear_causal_gb300 import binding as gb, synth
    shape = synth.PRODUCTION
    cfg = gb.make_config(16, 32, 128, 128, 4, True, 1e-6, "bf16")
    n_in = len(steps)
    qkv = torch.stack([_to_dev(s["qkv"], dev) for s in steps])
    gate = torch.stack([_to_dev(s["gate"], dev) for s in steps])
    beta = torch.stack([_to_dev(s["beta"], dev) for s in steps])
    w = _to_dev(st["conv_weight"], dev)
    per_step = decode_bytes(shape, B_DECODE)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    R = max(2, math.ceil(2 * l2 / per_step))
    S = [_to_dev(st["ssm_state"], dev) for _ in range(R)]
    conv = [_to_dev(st["conv_state"], dev) for _ in range(R)]
    out = torch.empty(B_DECODE, 32, 128, device=dev)
    stream = torch.cuda.current_stream()

    def step(i):
        j, r = i % n_in, i % R
        gb.gdn_forward_decode(cfg, B_DECODE, qkv[j], w, gate[j], beta[j], conv[r], S[r], out)

    for i in range(args.warmup):
        step(i)
    # untimed soak (at most args.soak launches, ~40 ms) so clocks settle under this load
    torch.cuda.synchronize()
    for i in range(args.soak):
        step(i)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ms = _max_over_ranks(dist, e0.elapsed_time(e1), dev)
    value = _job_value(B_DECODE * args.steps, world, ms)
    launch_us = ms * 1e3 / args.steps

    if args.no_e2e:
        return dict(ms=ms, value=value, launch_us=launch_us, bytes=per_step, rotation=R, e2e=None,
                     inputs=dict(steps=steps, state=st))
    # End to end through the public binding, pipelined the way a serving loop runs it: each
    # step's inputs (one packed pinned buffer) are copied in on an H2D stream and its output
    # copied back to pinned memory on a D2H stream; two device buffer sets alternate, so the
    # copies of neighbouring steps overlap the kernel.  Every step still moves its own bytes.
    nq, ng = steps[0]["qkv"].size * 2, steps[0]["gate"].size * 4
    nbytes = nq + 2 * ng
    h_in = []
    for s_ in steps:
        packed = np.concatenate([np.ascontiguousarray(s_["qkv"]).view(np.uint8).ravel(),
                                 np.ascontiguousarray(s_["gate"], dtype=np.float32).view(np.uint8).ravel(),
                                 np.ascontiguousarray(s_["beta"], dtype=np.float32).view(np.uint8).ravel()])
        h_in.append(torch.from_numpy(packed).pin_memory())
    d_in = [torch.empty(nbytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    views = [(b[:nq].view(torch.bfloat16).view(qkv[0].shape), b[nq:nq + ng].view(torch.float32).view(gate[0].shape),
              b[nq + ng:].view(torch.float32).view(beta[0].shape)) for b in d_in]
    d_out = [torch.empty_like(out) for _ in range(2)]
    h_out = [torch.empty(B_DECODE, 32, 128).pin_memory() for _ in range(2)]
    s_h2d, s_d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    # the C-ABI call itself, its pointers marshalled once (the binding's per-call tensor checks
    # would otherwise take as long as the kernel on this host)
    import ctypes
    abi, cfg_ref, sh = gb.load().gdn_forward_decode, ctypes.byref(cfg), stream.cuda_stream
    ptrs = {(k, r): (views[k][0].data_ptr(), w.data_ptr(), views[k][1].data_ptr(), views[k][2].data_ptr(),
                     conv[r].data_ptr(), S[r].data_ptr(), d_out[k].data_ptr()) for k in range(2) for r in range(R)}
    ev_in = [torch.cuda.Event() for _ in range(2)]   # inputs of set k landed
    ev_k = [torch.cuda.Event() for _ in range(2)]    # the kernel on set k has finished
    ev_out = [torch.cuda.Event() for _ in range(2)]  # output of set k is back on the host
    used = [False, False]
    rt = _cudart_calls()
    if rt is not None:
        # the same step with the CUDA runtime's copy, event and wait calls made directly (the
        # runtime already loaded in this process): torch's Python dispatch of those eight calls
        # per step would take about as long as the kernel on this host
        memcpy, record, wait, create, devptr = rt
        evs = []
        for _ in range(6):
            h = ctypes.c_void_p()
            if create(ctypes.byref(h), 2):  # cudaEventDisableTiming
                raise RuntimeError("cudaEventCreateWithFlags failed")
            evs.append(h)
        c_in, c_k, c_out = evs[0:2], evs[2:4], evs[4:6]
        sm, s1, s2 = ctypes.c_void_p(sh), ctypes.c_void_p(s_h2d.cuda_stream), ctypes.c_void_p(s_d2h.cuda_stream)
        hin = [h.data_ptr() for h in h_in]
        din, dout, hout = [b.data_ptr() for b in d_in], [o.data_ptr() for o in d_out], [o.data_ptr() for o in h_out]
        nout = h_out[0].numel() * 4

        def e2e_step(i):
            j, r, k = i % n_in, i % R, i & 1
            if used[k]:
                wait(s1, c_k[k], 0)  # the kernel two steps back is done with d_in[k]
            e = memcpy(din[k], hin[j], nbytes, 1, s1) or record(c_in[k], s1) or wait(sm, c_in[k], 0)
            if not e and used[k]:
                e = wait(sm, c_out[k], 0)  # d_out[k] has been read back
            if e:
                raise RuntimeError(f"CUDA runtime error {e} in the e2e step")
            rc = abi(cfg_ref, B_DECODE, *ptrs[(k, r)], sh)
            if rc:
                raise RuntimeError(f"gdn_forward_decode: {gb.gdn_status_string(rc)}")
            e = record(c_k[k], sm) or wait(s2, c_k[k], 0) or memcpy(hout[k], dout[k], nout, 2, s2) or record(c_out[k], s2)
            if e:
                raise RuntimeError(f"CUDA runtime error {e} in the e2e step")
            used[k] = True

        def drain():
            for k in range(2):
                if used[k]:
                    wait(sm, c_out[k], 0)
    else:
        def drain():
            for k in range(2):
                if used[k]:
                    stream.wait_event(ev_out[k])

    def e2e_step_torch(i):
        j, r, k = i % n_in, i % R, i & 1
        if used[k]:
            s_h2d.wait_event(ev_k[k])  # the kernel two steps back is done with d_in[k]
        with torch.cuda.stream(s_h2d):
            d_in[k].copy_(h_in[j], non_blocking=True)
            ev_in[k].record(s_h2d)
        stream.wait_event(ev_in[k])
        if used[k]:
            stream.wait_event(ev_out[k])  # d_out[k] has been read back
        rc = abi(cfg_ref, B_DECODE, *ptrs[(k, r)], sh)
        if rc:
            raise RuntimeError(f"gdn_forward_decode: {gb.gdn_status_string(rc)}")
        ev_k[k].record(stream)
        s_d2h.wait_event(ev_k[k])
        with torch.cuda.stream(s_d2h):
            h_out[k].copy_(d_out[k], non_blocking=True)
            ev_out[k].record(s_d2h)
        used[k] = True

    if rt is None:
        e2e_step = e2e_step_torch
    for i in range(args.warmup):
        e2e_step(i)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    s_h2d.wait_event(e0)
    for i in range(args.steps):
        e2e_step(i)
    drain()
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = _max_over_ranks(dist, e0.elapsed_time(e1), dev)
    h2d = nbytes
    d2h = h_out[0].numel() * 4
    # The same steps with the kernel reading each step's inputs from, and writing its output
    # to, the pinned host buffers themselves (NVLink-C2C; device addresses of the pinned
    # memory from cudaHostGetDevicePointer): every step still moves its own bytes between
    # host and device, with no copy, event or wait between consecutive launches.
    ms_zc = None
    if rt is not None:
        def dptr(t):
            p_ = ctypes.c_void_p()
            return None if devptr(ctypes.byref(p_), ctypes.c_void_p(t.data_ptr()), 0) else p_.value
        zin, zout = [dptr(h) for h in h_in], [dptr(h) for h in h_out]
        if all(p_ is not None for p_ in zin + zout):
            zptrs = {(j, k, r): (zin[j], w.data_ptr(), zin[j] + nq, zin[j] + nq + ng, conv[r].data_ptr(),
                                 S[r].data_ptr(), zout[k]) for j in range(n_in) for k in range(2) for r in range(R)}

            def zstep(i):
                rc = abi(cfg_ref, B_DECODE, *zptrs[(i % n_in, i & 1, i % R)], sh)
                if rc:
                    raise RuntimeError(f"gdn_forward_decode: {gb.gdn_status_string(rc)}")

            torch.cuda.synchronize()
            for i in range(args.warmup):
                zstep(i)
            if dist:
                dist.barrier()
            torch.cuda.synchronize()
            e0.record(stream)
            for i in range(args.steps):
                zstep(i)
            e1.record(stream)
            torch.cuda.synchronize()
            ms_zc = _max_over_ranks(dist, e0.elapsed_time(e1), dev)
    return dict(ms=ms, value=value, launch_us=launch_us, bytes=per_step, rotation=R,
                e2e=None if args.no_e2e else dict(value=_job_value(B_DECODE * args.steps, world, ms_e2e), unit="tokens/s",
                         h2d_bytes_per_step=h2d,
                         d2h_bytes_per_step=d2h, overlap="H2D and D2H streams, two buffer sets: copies of "
                         "neighbouring steps overlap the kernel",
                         host_calls="CUDA runtime via ctypes" if rt is not None else "torch",
                         zero_copy_value=None if ms_zc is None else _job_value(B_DECODE * args.steps, world, ms_zc)),
                inputs=dict(steps=steps, state=st))


def _cudart_calls():
    """cudaMemcpyAsync, cudaEventRecord, cudaStreamWaitEvent and cudaEventCreateWithFlags of the
    CUDA runtime this process has loaded (torch's and the library's), or None."""
    import ctypes
    try:
        rt = ctypes.CDLL("libcudart.so.13")
    except OSError:
        return None
    vp, c = ctypes.c_void_p, ctypes
    memcpy, record, wait, create = rt.cudaMemcpyAsync, rt.cudaEventRecord, rt.cudaStreamWaitEvent, rt.cudaEventCreateWithFlags
    memcpy.argtypes, memcpy.restype = [vp, vp, c.c_size_t, c.c_int, vp], c.c_int
    record.argtypes, record.restype = [vp, vp], c.c_int
    wait.argtypes, wait.restype = [vp, vp, c.c_uint], c.c_int
    create.argtypes, create.restype = [c.POINTER(vp), c.c_uint], c.c_int
    devptr = rt.cudaHostGetDevicePointer
    devptr.argtypes, devptr.restype = [c.POINTER(vp), vp, c.c_uint], c.c_int
    return memcpy, record, wait, create, devptr


def _time_calls(fn, reps, flush):
    """Device time of one call of fn per repetition, L2 flushed before each.  The flush
    and a short device-side spin are queued ahead of the start event, so the host's
    argument marshalling and launch of fn overlap them and stay out of the timed span."""
    import torch
    times = []
    for _ in range(reps):
        torch.cuda.synchronize()
        flush()
        torch.cuda._sleep(400_000)  # ~0.2 ms of device time at 2 GHz
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    return statistics.median(times), times


def run_decode_raw_gates(dev, st, steps, n_steps=128):
    """Decode B=64 with the gate parameterisation done in the kernel (config carries
    A_log and dt_bias; the gate/beta inputs are the raw projections).  Back-to-back
    steps over 2 rotating state sets, like the headline; returns ms per step."""
    import torch
    from gated_deltanet_linear_causal_gb300 import binding as gb, synth
    n_in = len(steps)
    raw = synth.raw_gates(7, (n_in, B_DECODE), 32)
    cfg = gb.make_config(16, 32, 128, 128, 4, True, 1e-6, "bf16", A_log=_to_dev(raw["A_log"], dev),
                         dt_bias=_to_dev(raw["dt_bias"], dev))
    qkv = torch.stack([_to_dev(s["qkv"], dev) for s in steps])
    a, b = _to_dev(raw["a"], dev), _to_dev(raw["b"], dev)
    w = _to_dev(st["conv_weight"], dev)
    S = [_to_dev(st["ssm_state"], dev) for _ in range(2)]
    conv = [_to_dev(st["conv_state"], dev) for _ in range(2)]
    out = torch.empty(B_DECODE, 32, 128, device=dev)

    def step(i):
        j, r = i % n_in, i % 2
        gb.gdn_forward_decode(cfg, B_DECODE, qkv[j], w, a[j], b[j], conv[r], S[r], out)

    for i in range(8):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(n_steps):
        step(i)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n_steps


def run_decode_gated(dev, st, steps, n_steps=128):
    """Decode B=64 with the gated RMSNorm (section 2) fused into the output epilogue:
    bf16 z in, bf16 y out instead of the fp32 output.  Returns ms per step."""
    import torch
    from gated_deltanet_linear_causal_gb300 import binding as gb, synth
    n_in = len(steps)
    d = synth.Draw(8)
    cfg = gb.make_config(16, 32, 128, 128, 4, True, 1e-6, "bf16")
    qkv = torch.stack([_to_dev(s["qkv"], dev) for s in steps])
    gate = torch.stack([_to_dev(s["gate"], dev) for s in steps])
    beta = torch.stack([_to_dev(s["beta"], dev) for s in steps])
    z = _to_dev(d.bf16("z", (n_in, B_DECODE, 32, 128)), dev)
    w_n = _to_dev(d.f32("norm_w", (128,), 1.0, 0.3), dev)
    w = _to_dev(st["conv_weight"], dev)
    S = [_to_dev(st["ssm_state"], dev) for _ in range(2)]
    conv = [_to_dev(st["conv_state"], dev) for _ in range(2)]
    y = torch.empty(B_DECODE, 32, 128, dtype=torch.bfloat16, device=dev)

    out = torch.empty(B_DECODE, 32, 128, device=dev)

    def step(i):
        j, r = i % n_in, i % 2
        gb.gdn_forward_decode_gated(cfg, B_DECODE, qkv[j], w, gate[j], beta[j], conv[r], S[r], z[j], w_n, 1e-6, y)

    def step_unfused(i):  # the same through gdn_forward_decode, then the standalone norm
        j, r = i % n_in, i % 2
        gb.gdn_forward_decode(cfg, B_DECODE, qkv[j], w, gate[j], beta[j], conv[r], S[r], out)
        gb.gdn_gated_rmsnorm(cfg, B_DECODE * 32, out, z[j], w_n, 1e-6, y)

    res = []
    for fn in (step, step_unfused):
        for i in range(8):
            fn(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(n_steps):
            fn(i)
        e1.record()
        torch.cuda.synchronize()
        res.append(e0.elapsed_time(e1) / n_steps)
    return res


def run_prefill(dev, x, variant, reps=20):
    import numpy as np
    import torch
    from gated_deltanet_linear_causal_gb300 import binding as gb, synth
    shape = x["shape"]
    cfg = gb.make_config(shape.num_k_heads, shape.num_v_heads, shape.head_k_dim, shape.head_v_dim, 4, True, 1e-6,
                         "bf16")
    cu = x["cu_seqlens"]
    N, T = len(cu) - 1, int(cu[-1])
    cu_d = _to_dev(cu, dev)
    qkv, w = _to_dev(x["qkv"], dev), _to_dev(x["conv_weight"], dev)
    gate, beta = _to_dev(x["gate"], dev), _to_dev(x["beta"], dev)
    conv0, S0 = _to_dev(x["conv_state"], dev), _to_dev(x["ssm_state"], dev)
    conv, S = conv0.clone(), S0.clone()
    out = torch.empty(T, shape.num_v_heads, shape.head_v_dim, device=dev)
    ws = torch.empty(max(1, gb.gdn_prefill_workspace_size(cfg, N, T, variant)), dtype=torch.uint8, device=dev)
    scratch = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def flush():  # restore the initial states and push the L2 out (256 MiB write)
        conv.copy_(conv0)
        S.copy_(S0)
        scratch.zero_()

    def call():
        gb.gdn_forward_prefill(cfg, N, cu_d, cu, qkv, w, gate, beta, conv, S, out, variant, ws)

    call()
    med, times = _time_calls(call, reps, flush)
    return med, times


def run_prefill_gated(dev, x, variant, reps=20):
    """The prefill with the gated RMSNorm fused (bf16 z in, bf16 y out), and the same
    through gdn_forward_prefill then gdn_gated_rmsnorm; returns both median times."""
    import torch
    from gated_deltanet_linear_causal_gb300 import binding as gb, synth
    shape = x["shape"]
    cfg = gb.make_config(shape.num_k_heads, shape.num_v_heads, shape.head_k_dim, shape.head_v_dim, 4, True, 1e-6,
                         "bf16")
    cu = x["cu_seqlens"]
    N, T = len(cu) - 1, int(cu[-1])
    H, dv = shape.num_v_heads, shape.head_v_dim
    d = synth.Draw(9)
    cu_d = _to_dev(cu, dev)
    qkv, w = _to_dev(x["qkv"], dev), _to_dev(x["conv_weight"], dev)
    gate, beta = _to_dev(x["gate"], dev), _to_dev(x["beta"], dev)
    conv0, S0 = _to_dev(x["conv_state"], dev), _to_dev(x["ssm_state"], dev)
    conv, S = conv0.clone(), S0.clone()
    z = _to_dev(d.bf16("z", (T, H, dv)), dev)
    w_n = _to_dev(d.f32("norm_w", (dv,), 1.0, 0.3), dev)
    y = torch.empty(T, H, dv, dtype=torch.bfloat16, device=dev)
    out = torch.empty(T, H, dv, device=dev)
    ws = torch.empty(max(1, gb.gdn_prefill_workspace_size(cfg, N, T, variant)), dtype=torch.uint8, device=dev)
    scratch = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def flush():
        conv.copy_(conv0)
        S.copy_(S0)
        scratch.zero_()

    def fused():
        gb.gdn_forward_prefill_gated(cfg, N, cu_d, cu, qkv, w, gate, beta, conv, S, z, w_n, 1e-6, y, variant, ws)

    def unfused():
        gb.gdn_forward_prefill(cfg, N, cu_d, cu, qkv, w, gate, beta, conv, S, out, variant, ws)
        gb.gdn_gated_rmsnorm(cfg, T * H, out, z, w_n, 1e-6, y)

    res = []
    for fn in (fused, unfused):
        fn()
        res.append(_time_calls(fn, reps, flush))
    return res


def run_verify(dev, x, reps=20):
    import torch
    from gated_deltanet_linear_causal_gb300 import binding as gb
    shape = x["shape"]
    B, L = x["qkv"].shape[0], x["qkv"].shape[2]
    cfg = gb.make_config(16, 32, 128, 128, 4, True, 1e-6, "bf16")
    d = {k: _to_dev(x[k], dev) for k in ("qkv", "conv_weight", "gate", "beta", "conv_state", "ssm_state", "accepted")}
    csnap = torch.empty(B, L, shape.D, 3, dtype=torch.bfloat16, device=dev)
    ssnap = torch.empty(B, L, 32, 128, 128, device=dev)
    out = torch.empty(B, L, 32, 128, device=dev)
    scratch = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def verify():
        gb.gdn_forward_verify(cfg, B, L, d["qkv"], d["conv_weight"], d["gate"], d["beta"], d["conv_state"],
                              d["ssm_state"], csnap, ssnap, out)

    def commit():
        gb.gdn_verify_commit(cfg, B, L, d["accepted"], csnap, ssnap, d["conv_state"], d["ssm_state"])

    verify()
    mv, tv = _time_calls(verify, reps, lambda: scratch.zero_())
    mc, _ = _time_calls(commit, reps, lambda: (verify(), scratch.zero_()))
    return mv, mc, tv


def _env(dev):
    """The device and software the numbers were taken on."""
    import torch
    p = torch.cuda.get_device_properties(dev)
    env = {"gpu": p.name, "sm": f"sm_{p.major}{p.minor}", "sms": p.multi_processor_count,
           "torch": torch.__version__, "cuda_runtime": torch.version.cuda, "driver": None}
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader", "-i",
                              str(dev.index)], capture_output=True, text=True, timeout=10)
        env["driver"] = out.stdout.strip() or None
    except (OSError, subprocess.SubprocessError):
        pass
    return env


def _spread(times):
    """Relative spread of the repetitions: max / min - 1."""
    return round(max(times) / min(times) - 1.0, 4)


# ---------------------------------------------------------------------------
# fp64 oracle on the host cores
# ---------------------------------------------------------------------------

def _host_cpu():
    """The host the oracle runs on: its logical core count and CPU model."""
    model = None
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except OSError:
        pass
    if not model:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.strip().lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    import platform
    return {"host_cores": os.cpu_count(), "cpu_model": model or platform.processor() or platform.machine()}


def oracle_decode_rate(steps, state, budget_s, max_steps):
    """Oracle decode steps of the B=64 workload (all sequences, all heads) until the
    time budget is spent; returns (tokens/s, sample description)."""
    import oracle
    from gated_deltanet_linear_causal_gb300 import synth
    shape = synth.PRODUCTION
    ocfg = oracle.Cfg(16, 32, 128, 128, 4, True, 1e-6)
    conv = synth.as_f64(state["conv_state"], "bf16")
    S = state["ssm_state"].astype("float64")
    w = synth.as_f64(state["conv_weight"], "bf16")
    t0 = time.perf_counter()
    tokens, n = 0, 0
    seqs_per_chunk = 8
    while n < max_steps:
        s = steps[n % len(steps)]
        qkv = synth.as_f64(s["qkv"], "bf16")
        for b0 in range(0, B_DECODE, seqs_per_chunk):
            idx = list(range(b0, b0 + seqs_per_chunk))
            _, c_new, S_new = oracle.decode(ocfg, qkv, w, s["gate"], s["beta"], conv, S, batch_index=idx)
            conv[idx], S[idx] = c_new, S_new
            tokens += len(idx)
            if time.perf_counter() - t0 > budget_s:
                break
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return tokens / dt, f"{tokens} decode tokens ({n} step(s) of the B=64 workload, all 32 heads) in {dt:.1f} s"


# ---------------------------------------------------------------------------

SECONDARIES = ("prefill_chunked", "prefill_resident", "prefill_gated_norm", "decode_raw_gates", "decode_gated_norm",
               "verify")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-secondary", action="store_true", help="headline decode only")
    ap.add_argument("--soak", type=int, default=500, help="untimed decode launches before the timed region")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--only", default="", help="comma list of secondaries to run (default all): " + ", ".join(SECONDARIES))
    args = ap.parse_args()
    bad = [n for n in args.only.split(",") if n and n not in SECONDARIES]
    if bad:
        ap.error(f"unknown secondaries {bad}; choose from {SECONDARIES}")
    args.warmup = max(args.warmup, 3)

    if args.impl == "reference":
        return main_reference(args)

    import torch
    dist, rank, world = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from gated_deltanet_linear_causal_gb300 import binding as gb, synth
    gb.load()
    peaks = _peaks()
    secondary = world == 1 and not args.no_secondary
    st, steps = decode_inputs(args, rank)
    if secondary:  # host-side input generation happens before the GPU-timed phases
        x_long, x_var, x_ver = synth.long_prefill(seed=3), synth.varlen_prefill(seed=4), synth.verify_block(seed=5)
    clocks = ClockSampler(dev.index)  # samples across the GPU phases of this run
    clocks.start()
    dec = run_decode(args, dev, dist, rank, world, st, steps)
    sec = {}
    only = set(n for n in args.only.split(",") if n) or set(SECONDARIES)
    if secondary and rank == 0:
        shape = synth.PRODUCTION
        chunk_sources = ["gdn_chunked.cu", "gdn_common.cuh", "gdn_tma.cuh", "gdn_umma.cuh"]
        for name, variant in (("chunked", gb.GDN_PREFILL_CHUNKED), ("resident", gb.GDN_PREFILL_RESIDENT)):
            if "prefill_" + name not in only:
                continue
            key = "" if name == "chunked" else "_resident"
            for label, x, rand in (("prefill_L8192", x_long, False), ("prefill_varlen16", x_var, True)):
                med, times = run_prefill(dev, x, variant)
                cu = x["cu_seqlens"]
                T = int(cu[-1])
                nb = prefill_bytes(shape, cu, rand)
                e = {"variant": name, "tokens": T, "tokens_per_s": round(T / (med / 1e3), 1), "ms": round(med, 4),
                     "reps": len(times), "spread": _spread(times),
                     "hbm_frac": round(nb / (med / 1e3) / 1e9 / peaks["hbm_gbs"], 4), "algorithmic_bytes": nb,
                     "cold_l2": True}
                if name == "chunked":
                    alg, issued = chunked_tensor_flops(shape, cu)
                    r = prefill_roofline(nb, issued, med, peaks)
                    e.update(algorithmic_tensor_flops=alg, issued_tensor_flops=issued, roofline=r,
                             roofline_frac=r["frac"],
                             traffic=_traffic(label.replace("prefill_", "prefill_chunked_"), chunk_sources,
                                              "chunked_prefill_L8192.json", "dram_bytes_per_call")
                             if label == "prefill_L8192" else None)
                else:
                    e["roofline_frac"] = e["hbm_frac"]  # bound by its serial chain; reported against HBM
                sec[label + key] = e
        for name, variant in (("chunked", gb.GDN_PREFILL_CHUNKED), ("resident", gb.GDN_PREFILL_RESIDENT)):
            if "prefill_gated_norm" not in only:
                break
            (mf, tf), (mu, _) = run_prefill_gated(dev, x_long, variant)
            key = "" if name == "chunked" else "_resident"
            sec["prefill_L8192_gated_norm" + key] = {
                "variant": name, "tokens_per_s": round(8192 / (mf / 1e3), 1), "ms": round(mf, 4), "reps": len(tf),
                "spread": _spread(tf), "ms_prefill_then_norm_kernel": round(mu, 4), "cold_l2": True,
                "note": "gated RMSNorm fused into the output epilogue (clusters exchange the rows' sums of squares): "
                        "bf16 z in, bf16 y out, no fp32 output written"}
        if "decode_raw_gates" in only:
            ms = run_decode_raw_gates(dev, st, steps)
            nb = decode_bytes(shape, B_DECODE) + 2 * 32 * 4
            sec["decode_B64_raw_gates"] = {"tokens_per_s": round(B_DECODE / (ms / 1e3), 1), "ms": round(ms, 5),
                                           "roofline_frac": round(nb / (ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                                           "algorithmic_bytes": nb,
                                           "note": "gate = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b) in the kernel"}
        if "decode_gated_norm" in only:
            ms, ms_unfused = run_decode_gated(dev, st, steps)
            nb = decode_bytes(shape, B_DECODE) - B_DECODE * 32 * 128 * 4 + 2 * B_DECODE * 32 * 128 * 2 + 128 * 4
            sec["decode_B64_gated_norm"] = {"tokens_per_s": round(B_DECODE / (ms / 1e3), 1), "ms": round(ms, 5),
                                            "roofline_frac": round(nb / (ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                                            "algorithmic_bytes": nb, "ms_decode_then_norm_kernel": round(ms_unfused, 5),
                                            "note": "gated RMSNorm fused: bf16 z in, bf16 y out"}
        if "verify" in only:
            mv, mc, tv = run_verify(dev, x_ver)
            nb = verify_bytes(shape, 32, 4)
            sec["verify_B32_L4"] = {"tokens_per_s": round(128 / (mv / 1e3), 1), "ms": round(mv, 4), "reps": len(tv),
                                    "spread": _spread(tv),
                                    "roofline_frac": round(nb / (mv / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                                    "algorithmic_bytes": nb, "commit_ms": round(mc, 4), "cold_l2": True}
    clk = clocks.stop()
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    achieved = dec["bytes"] / (dec["launch_us"] * 1e-6) / 1e9
    sources = ["gdn_stream.cu", "gdn_common.cuh", "gdn_tma.cuh"]
    line = {
        "metric": METRIC, "value": round(dec["value"], 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dec["ms"] / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "decode B=64, H_k=16, H_v=32, d_k=d_v=128, K=4, bf16 qkv, fp32 state, "
                               "fresh seeded inputs per step",
                   "global_batch": B_DECODE * world, "seq_len": 1, "parallelism": f"replicas{world}",
                   "io": "bf16", "l2": f"inputs larger than L2: {dec['rotation']} rotating state sets of "
                                         f"{dec['bytes'] / 1e6:.1f} MB per step"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": _traffic("decode_b64", sources),
                     "kernel": "stream_kernel<bf16,128,in_place>", "algorithmic_bytes_per_launch": dec["bytes"],
                     "launch_us": round(dec["launch_us"], 2), "peak_source": peaks["source"]},
        "e2e": dec["e2e"], "gpu_launches": args.steps, "clocks": clk, "env": _env(dev),
    }
    if world == 1 and args.cpu_budget > 0:
        v, sample = oracle_decode_rate(dec["inputs"]["steps"], dec["inputs"]["state"], args.cpu_budget, args.steps)
        line["cpu_baseline"] = {"value": round(v, 2), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                "sample": sample, **_host_cpu()}
    if sec:
        line["secondary"] = sec
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main_reference(args):
    """The fp64 oracle, single-threaded, on this host's cores, on the decode workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from gated_deltanet_linear_causal_gb300 import synth
    import oracle
    oracle.build()
    st = synth.decode_state(2, B_DECODE, synth.PRODUCTION)
    steps = [synth.decode_step(2, s, B_DECODE, synth.PRODUCTION) for s in range(4)]
    budget = max(2.0, min(args.cpu_budget, 8.0))
    t0 = time.perf_counter()
    v, sample = oracle_decode_rate(steps, st, budget, max(1, args.steps))
    total = time.perf_counter() - t0
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 2), "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(B_DECODE / v * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "decode B=64, H_k=16, H_v=32, d_k=d_v=128, K=4, bf16 qkv (fp64 oracle)",
                       "global_batch": B_DECODE, "seq_len": 1, "parallelism": "host, 1 thread"},
            "cpu_baseline": {"value": round(v, 2), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": sample, **_host_cpu()},
            "e2e": {"value": round(v, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(total, 2)}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
