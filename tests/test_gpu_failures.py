"""Failure detection on the GPU without faulting it: bad group offsets and a
wait that runs out each set a bit of the sticky device status word, the
affected kernel skips its work and returns, and the context stays usable."""
import numpy as np
import pytest
import torch

from tests import harness as H
from workloads import WORKLOADS, make_inputs, scaled

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

MOE_DEV_BAD_OFFSETS, MOE_DEV_TIMEOUT = 0x1, 0x4


def test_wait_timeout_sets_status_and_context_survives():
    import moe_expert_mlp_gb300 as m
    assert m.moe_read_device_status(clear=True) == 0
    m._lib.moe_selftest_wait_timeout(50000)            # 50 ms, nothing completes the phase
    assert m.moe_read_device_status(clear=True) & MOE_DEV_TIMEOUT
    assert m.moe_read_device_status(clear=False) == 0
    # the context still runs real work afterwards
    wl = scaled(WORKLOADS["bf16_t4096_e64"], T=256, E=4, k=2, d=128, F=64)
    layer = H.run_gpu_routed(wl, make_inputs(wl))
    assert m.moe_read_device_status() == 0
    assert torch.isfinite(layer.out.float()).all()


def test_grid_barrier_timeout_sets_status_and_context_survives():
    """The fused router's grid-wide barrier: a CTA waiting for an arrival
    that never comes gives up after its limit, sets the timeout bit and
    returns; the fused router then still runs correctly."""
    import moe_expert_mlp_gb300 as m
    assert m.moe_read_device_status(clear=True) == 0
    m._lib.moe_selftest_grid_wait_timeout(50000)       # 50 ms, the second arrival never comes
    assert m.moe_read_device_status(clear=True) & MOE_DEV_TIMEOUT
    assert m.moe_read_device_status(clear=False) == 0
    wl = scaled(WORKLOADS["bf16_t4096_e64"], T=300, E=8, k=2, d=128, F=64)
    inp = make_inputs(wl, with_weights=False)
    layer = H.make_layer(wl)
    wr = torch.randn((wl.E, wl.d), device="cuda").to(torch.bfloat16)
    layer.route_fused(H.bits_to_dev(inp["x"]), wr)
    torch.cuda.synchronize()
    assert m.moe_read_device_status() == 0
    assert int(layer.counts.sum()) == wl.T * wl.k


def test_inconsistent_offsets_are_detected_and_skipped():
    import moe_expert_mlp_gb300 as m
    wl = scaled(WORKLOADS["dsv3_r16384_e32"], R=300, E=4, d=128, F=64, zipf_empty=0)
    inp = make_inputs(wl)
    layer, _ = H.run_both_direct(wl, inp)
    assert m.moe_read_device_status() == 0
    y_before = layer.y.clone()
    good = layer.padded_offsets.clone()
    bad = good.clone()
    bad[2] = bad[1] + 64                               # not a multiple of 128: inconsistent
    layer.padded_offsets.copy_(bad)
    layer.y.fill_(7.0)
    layer.mlp_forward()
    torch.cuda.synchronize()
    assert m.moe_read_device_status(clear=True) & MOE_DEV_BAD_OFFSETS
    assert torch.all(layer.y == 7.0)                   # FC2 skipped its work entirely
    layer.padded_offsets.copy_(good)
    layer.mlp_forward()
    torch.cuda.synchronize()
    assert m.moe_read_device_status() == 0
    assert torch.equal(layer.y, y_before)
