"""Library behaviour that is not arithmetic: state init, asynchrony, device errors."""
import time

import numpy as np
import pytest
import torch

from gated_deltanet_linear_causal_gb300 import binding as gb
from gated_deltanet_linear_causal_gb300 import synth
from gdn_testutil import configs, device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_conv_state_init_zeroes_both_states(io):
    dev = device()
    cfg, _ = configs(synth.Shape(2, 4, 32, 32, 3), io)
    conv = torch.full((5, cfg.D, 2), 7.0, dtype=cfg.torch_dtype, device=dev)
    S = torch.full((5, 4, 32, 32), 3.0, device=dev)
    gb.gdn_conv_state_init(cfg, 5, conv, S)
    torch.cuda.synchronize()
    assert bool((conv == 0).all()) and bool((S == 0).all())
    # an offset view (unaligned start) is zeroed exactly over its own range
    buf = torch.full((1 + 5 * cfg.D * 2,), 9.0, dtype=cfg.torch_dtype, device=dev)
    gb.gdn_conv_state_init(cfg, 5, buf[1:], None)
    torch.cuda.synchronize()
    assert float(buf[0]) == 9.0 and bool((buf[1:] == 0).all())


def test_calls_do_not_block_the_host():
    """A call only enqueues work: behind a ~0.2 s device sleep it still returns at once
    (isolated vs pipelined timing, as the mlxcel benchmark notes use to catch host syncs)."""
    dev = device()
    shape = synth.PRODUCTION
    cfg, _ = configs(shape, "bf16")
    B = 8
    st = synth.decode_state(2, B, shape)
    d = synth.decode_step(2, 0, B, shape)
    from gdn_testutil import to_dev
    args = [to_dev(d["qkv"], dev), to_dev(st["conv_weight"], dev), to_dev(d["gate"], dev), to_dev(d["beta"], dev),
            to_dev(st["conv_state"], dev), to_dev(st["ssm_state"], dev),
            torch.empty(B, 32, 128, device=dev)]
    gb.gdn_forward_decode(cfg, B, *args)  # warm: module load, attributes
    torch.cuda.synchronize()
    torch.cuda._sleep(400_000_000)
    t0 = time.perf_counter()
    gb.gdn_forward_decode(cfg, B, *args)
    dt = time.perf_counter() - t0
    torch.cuda.synchronize()
    assert dt < 0.05, f"decode call took {dt:.3f} s on the host"


def test_errors_raise_before_launch():
    dev = device()
    cfg, _ = configs(synth.ORACLE_SCALE, "f32")
    t = torch.zeros(1 << 16, device=dev)
    with pytest.raises(ValueError):   # the binding sizes the workspace before calling
        gb.gdn_forward_prefill(cfg, 1, torch.tensor([0, 4], dtype=torch.int32, device=dev), np.array([0, 4], np.int32),
                               t, t, t, t, t, t, t, gb.GDN_PREFILL_RESIDENT, torch.empty(16, dtype=torch.uint8,
                                                                                        device=dev))
    with pytest.raises(gb.GdnError) as e:
        gb.gdn_forward_decode(cfg, 1, t[1:], t, t, t, t, t, t)  # qkv 4 bytes off 16-byte alignment
    assert e.value.status == 3
    with pytest.raises(gb.GdnError) as e:
        gb.gdn_forward_prefill(cfg, 2, torch.tensor([0, 4, 2], dtype=torch.int32, device=dev),
                               np.array([0, 4, 2], np.int32), t, t, t, t, t, t, t, gb.GDN_PREFILL_RESIDENT,
                               torch.empty(1 << 20, dtype=torch.uint8, device=dev))
    assert e.value.status == 5


def test_no_device_side_wait_gave_up():
    """No bounded wait of any kernel run so far in this process timed out."""
    device()
    assert gb.gdn_device_error() == 0
