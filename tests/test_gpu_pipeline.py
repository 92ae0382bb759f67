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
