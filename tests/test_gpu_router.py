"""Fused router (router GEMM with the top-k in its epilogue and the
permutation in the same cooperative launch) against the oracle.  The logits come from the tensor cores in fp32; they are checked
against the oracle's fp64 x W_r^T within the fp32 accumulation error, and
the selection -- an integer decision taken in floating point -- is checked
bit for bit against the oracle's routing applied to the kernel's own fp32
logits (both sides decide in the kernel's precision).  Offsets, the
permutation and x_perm then follow bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from tests import harness as H
from workloads import WORKLOADS, bf16_bits_to_f64, f32_to_bf16_bits, make_inputs, scaled

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

BASE = WORKLOADS["bf16_t4096_e64"]
CASES = {
    "tiny": (WORKLOADS["tiny_t256_e8"], False),
    "e64_k6_bias": (scaled(BASE, T=1000, d=512, F=128), True),
    "e40_k3_ragged": (scaled(BASE, T=777, E=40, k=3, d=320, F=64), True),
    "e200_k8": (scaled(BASE, T=300, E=200, k=8, d=256, F=64), False),
    # more 256-token chunks (157) than CTAs: the in-launch assignment loops
    "many_chunks": (scaled(BASE, T=40000, E=16, k=2, d=128, F=64), True),
    "one_token": (scaled(BASE, T=1, E=8, k=2, d=128, F=64), False),
}


@pytest.mark.parametrize("name", list(CASES))
def test_fused_router_matches_oracle(name):
    wl, with_bias = CASES[name]
    inp = make_inputs(wl, with_weights=False)
    rng = np.random.default_rng(7)
    wr_bits = f32_to_bf16_bits((rng.standard_normal((wl.E, wl.d)) / np.sqrt(wl.d)).astype(np.float32))
    bias = (rng.standard_normal(wl.E).astype(np.float32) * 0.5) if with_bias else None
    layer = H.make_layer(wl)
    x = H.bits_to_dev(inp["x"])
    logits = torch.zeros((wl.T, wl.E), dtype=torch.float32, device="cuda")
    layer.route_fused(x, H.bits_to_dev(wr_bits), torch.from_numpy(bias).cuda() if with_bias else None,
                      logits)
    torch.cuda.synchronize()
    from moe_expert_mlp_gb300 import moe_read_device_status
    assert moe_read_device_status() == 0
    # logits within the fp32 accumulation error of the exact product
    ref = bf16_bits_to_f64(inp["x"]) @ bf16_bits_to_f64(wr_bits).T
    lg = H.to_np(logits)
    H.assert_close("logits", lg, ref, rel=1e-5, abs_=1e-6)
    # routing decided on the kernel's fp32 logits
    topk_idx, topk_w, counts = oracle.route(lg, bias, wl.k)
    assert np.array_equal(H.to_np(layer.topk_idx)[:wl.T], topk_idx)
    H.assert_close("topk_w", H.to_np(layer.topk_w)[:wl.T], topk_w, rel=1e-5, abs_=1e-6)
    assert np.array_equal(H.to_np(layer.counts), counts)
    offsets, padded, tiles = oracle.group_offsets(counts, 128)
    assert np.array_equal(H.to_np(layer.offsets), offsets)
    assert np.array_equal(H.to_np(layer.padded_offsets), padded)
    assert np.array_equal(H.to_np(layer.tile_prefix), tiles)
    row_src, row_of = oracle.permute_index(topk_idx, wl.E, padded)
    R_pad = int(padded[-1])
    assert np.array_equal(H.to_np(layer.row_src)[:R_pad], row_src)
    assert np.array_equal(H.to_np(layer.row_of)[:wl.T], row_of)
    assert np.array_equal(H.to_np(layer.x_perm)[:R_pad],
                          oracle.gather_rows(bf16_bits_to_f64(inp["x"]), row_src))


def test_fused_router_equals_route_permute_on_its_logits():
    """The unfused path given the fused router's logits routes identically."""
    wl, _ = CASES["e64_k6_bias"]
    inp = make_inputs(wl, with_weights=False)
    rng = np.random.default_rng(8)
    wr = H.bits_to_dev(f32_to_bf16_bits(
        (rng.standard_normal((wl.E, wl.d)) / np.sqrt(wl.d)).astype(np.float32)))
    bias = torch.from_numpy(rng.standard_normal(wl.E).astype(np.float32)).cuda()
    x = H.bits_to_dev(inp["x"])
    logits = torch.zeros((wl.T, wl.E), dtype=torch.float32, device="cuda")
    fused = H.make_layer(wl)
    fused.route_fused(x, wr, bias, logits)
    plain = H.make_layer(wl)
    plain.route(x, logits, bias)
    torch.cuda.synchronize()
    for n in ("topk_idx", "counts", "padded_offsets", "row_src", "row_of"):
        assert torch.equal(getattr(fused, n), getattr(plain, n)), n
    assert torch.equal(fused.x_perm.view(torch.int16), plain.x_perm.view(torch.int16))
    assert torch.allclose(fused.topk_w, plain.topk_w, rtol=1e-6, atol=1e-7)


def test_fused_router_replays_in_a_cuda_graph():
    """The cooperative launch is captured in a CUDA graph; replays give the
    eager call's results bit for bit (the grid-barrier counter is zeroed by
    a memset node of the same graph before every launch)."""
    wl, _ = CASES["e40_k3_ragged"]
    inp = make_inputs(wl, with_weights=False)
    rng = np.random.default_rng(9)
    wr = H.bits_to_dev(f32_to_bf16_bits(
        (rng.standard_normal((wl.E, wl.d)) / np.sqrt(wl.d)).astype(np.float32)))
    bias = torch.from_numpy(rng.standard_normal(wl.E).astype(np.float32)).cuda()
    x = H.bits_to_dev(inp["x"])
    eager = H.make_layer(wl)
    eager.route_fused(x, wr, bias)
    torch.cuda.synchronize()
    layer = H.make_layer(wl)
    layer.route_fused(x, wr, bias)              # warm-up outside the capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            layer.route_fused(x, wr, bias, stream=s)
    for n in ("topk_idx", "counts", "padded_offsets", "row_src", "row_of", "x_perm"):
        getattr(layer, n).zero_()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    from moe_expert_mlp_gb300 import moe_read_device_status
    assert moe_read_device_status() == 0
    for n in ("topk_idx", "counts", "offsets", "padded_offsets", "tile_prefix", "row_src",
              "row_of"):
        assert torch.equal(getattr(layer, n), getattr(eager, n)), n
    assert torch.equal(layer.x_perm.view(torch.int16), eager.x_perm.view(torch.int16))
