"""HostStepPipeline: steps on host-resident batches with overlapped copies
give, step for step, the same results bit for bit as MoEExpertMLP.step with
in-line copies (the layer's kernels are deterministic)."""
import numpy as np
import pytest
import torch

from tests import harness as H
from workloads import WORKLOADS, make_inputs, scaled

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]


def test_pipeline_matches_serial_steps():
    from moe_expert_mlp_gb300.pipeline import HostStepPipeline
    wl = scaled(WORKLOADS["bf16_t4096_e64"], T=600, E=16, k=4, d=256, F=192)
    inp = make_inputs(wl)
    layer = H.make_layer(wl)
    H.load_layer_weights(layer, inp)
    bias = torch.from_numpy(inp["bias"]).cuda() if inp["bias"] is not None else None
    steps = []
    for seed in (1, 2, 3, 4):
        s = make_inputs(wl, seed=seed, with_weights=False)
        steps.append(dict(x=H.bits_to_dev(s["x"], "cpu").pin_memory(),
                          logits=torch.from_numpy(s["logits"]).pin_memory(),
                          dout=H.bits_to_dev(s["dout"], "cpu").pin_memory()))
    outs = [dict(out=torch.empty(layer.out.shape, dtype=layer.out.dtype).pin_memory(),
                 dx=torch.empty(layer.dx.shape, dtype=layer.dx.dtype).pin_memory(),
                 dlogits=torch.empty(layer.dlogits.shape, dtype=torch.float32).pin_memory())
            for _ in steps]
    HostStepPipeline(layer).run(steps, outs, bias)
    torch.cuda.synchronize()
    for st, o in zip(steps, outs):
        layer.step(st["x"].cuda(), st["logits"].cuda(), bias, st["dout"].cuda())
        torch.cuda.synchronize()
        assert torch.equal(o["out"].view(torch.int16), layer.out.cpu().view(torch.int16))
        assert torch.equal(o["dx"].view(torch.int16), layer.dx.cpu().view(torch.int16))
        assert torch.equal(o["dlogits"], layer.dlogits.cpu())
    # different batches gave different results (the buffers were not reused stale)
    assert not torch.equal(outs[0]["out"], outs[1]["out"])


def _grouped_serial(layer, x, dy, counts):
    """One grouped step with in-line copies into a freshly zeroed padded
    layout; returns the real rows of Y and dX_perm on the host."""
    from moe_expert_mlp_gb300.pipeline import GroupedHostStepPipeline
    segs = GroupedHostStepPipeline._segments(counts)
    layer.x_perm.zero_()
    layer.dy.zero_()
    for src, dst, m in segs:
        layer.x_perm[dst:dst + m].copy_(x[src:src + m])
        layer.dy[dst:dst + m].copy_(dy[src:src + m])
    layer.grouped_step(counts=counts.cuda())
    torch.cuda.synchronize()
    y = torch.cat([layer.y[dst:dst + m].cpu() for _, dst, m in segs])
    dx = torch.cat([layer.dx_perm[dst:dst + m].cpu() for _, dst, m in segs])
    return y, dx


@pytest.mark.parametrize("dtype,depth", [("bf16", 2), ("mxfp8", 2), ("bf16", 3)])
def test_grouped_pipeline_matches_serial_steps(dtype, depth):
    """GroupedHostStepPipeline (real rows only, moved group by group into the
    padded layout, two or three buffer sets in turn) == serial grouped steps, bit
    for bit, over four batches whose group sizes change after the second
    (the padded layout changes, old rows must not leak into padding)."""
    from moe_expert_mlp_gb300.pipeline import GroupedHostStepPipeline
    base = scaled(WORKLOADS["dsv3_r16384_e32"], R=900, E=7, d=256, F=192, zipf_empty=2)
    inp = make_inputs(base)
    sizes_a = inp["group_sizes"].astype(np.int32)
    sizes_b = np.roll(sizes_a, 3)                        # same R, different layout
    cap = max(int(sum((int(m) + 127) // 128 * 128 for m in s)) for s in (sizes_a, sizes_b))
    layer = H.make_layer(base, capacity=cap, dtype=dtype)
    H.load_layer_weights(layer, inp)
    R, d = int(sizes_a.sum()), base.d
    steps = []
    for i, seed in enumerate((1, 2, 3, 4)):
        s = make_inputs(scaled(base, seed=seed), with_weights=False)
        sizes = sizes_a if i < 2 else sizes_b
        steps.append(dict(x=H.bits_to_dev(s["x"][:R], "cpu").pin_memory(),
                          dy=H.bits_to_dev(s["dout"][:R], "cpu").pin_memory(),
                          counts=torch.from_numpy(sizes).pin_memory()))
    outs = [dict(y=torch.empty((R, d), dtype=torch.bfloat16).pin_memory(),
                 dx=torch.empty((R, d), dtype=torch.bfloat16).pin_memory()) for _ in steps]
    GroupedHostStepPipeline(layer, depth=depth).run(steps, outs)
    torch.cuda.synchronize()
    for st, o in zip(steps, outs):
        y, dx = _grouped_serial(layer, st["x"], st["dy"], st["counts"])
        assert torch.equal(o["y"].view(torch.int16), y.view(torch.int16))
        assert torch.equal(o["dx"].view(torch.int16), dx.view(torch.int16))
    assert not torch.equal(outs[0]["y"], outs[1]["y"])
