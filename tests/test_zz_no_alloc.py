"""moe_route_permute_noalloc: routing + permutation for callers that cannot
allocate device memory (their device memory belongs to a fixed pool of
their own, or their runtime forbids allocation after start-up).

The call keeps its scratch histogram in a static device array of the
library instead of a caller-provided workspace.  Through the C ABI it must
give the same results as the allocating moe_route_permute, on two calls in
a row (the shared array keeps the previous call's contents, so the second
call checks that the histogram is cleared before use).  This file is named
so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

from tests import harness as H
from workloads import WORKLOADS, make_inputs, scaled

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]


def _outputs(desc, T, E, k, d, dev):
    cap = desc.capacity
    i32, f32 = torch.int32, torch.float32
    return dict(
        topk_idx=torch.full((T, k), -7, dtype=i32, device=dev),
        topk_w=torch.full((T, k), -1.0, dtype=f32, device=dev),
        counts=torch.full((E,), -7, dtype=i32, device=dev),
        offsets=torch.full((E + 1,), -7, dtype=i32, device=dev),
        padded_offsets=torch.full((E + 1,), -7, dtype=i32, device=dev),
        tile_prefix=torch.full((E + 1,), -7, dtype=i32, device=dev),
        row_src=torch.full((cap,), -7, dtype=i32, device=dev),
        row_of=torch.full((T, k), -7, dtype=i32, device=dev),
        x_perm=torch.full((cap, d), 3.0, dtype=torch.bfloat16, device=dev),
    )


def _compare(got, ref):
    R_pad = int(ref["padded_offsets"][-1])
    for name in ("topk_idx", "counts", "offsets", "padded_offsets", "tile_prefix", "row_of"):
        assert torch.equal(got[name], ref[name]), name
    assert torch.equal(got["row_src"][:R_pad], ref["row_src"][:R_pad])
    assert torch.equal(got["x_perm"][:R_pad].view(torch.int16), ref["x_perm"][:R_pad].view(torch.int16))
    H.assert_close("topk_w", H.to_np(got["topk_w"]), H.to_np(ref["topk_w"]), rel=1e-5, abs_=1e-6)


def _routing_case(T, E, k, d):
    import moe_expert_mlp_gb300 as m
    from moe_expert_mlp_gb300 import _lib as L

    wl = scaled(WORKLOADS["bf16_t4096_e64"], T=max(T, 1), E=E, k=k, d=d, F=64)
    inp = make_inputs(wl, with_weights=False)
    dev = torch.device("cuda")
    desc = m.make_desc(T, E, k, d, 64)
    x = H.bits_to_dev(inp["x"])
    logits = torch.from_numpy(inp["logits"]).to(dev)
    bias = torch.from_numpy(inp["bias"]).to(dev)
    ref = _outputs(desc, max(T, 1), E, k, d, dev)
    ws = torch.zeros(max(m.moe_workspace_size(desc), 256), dtype=torch.uint8, device=dev)
    L.moe_route_permute(desc, logits, bias, x, ref["topk_idx"], ref["topk_w"], ref["counts"],
                        ref["offsets"], ref["padded_offsets"], ref["tile_prefix"], ref["row_src"],
                        ref["row_of"], ref["x_perm"], ws)
    torch.cuda.synchronize()
    return m, L, desc, logits, bias, x, ref


def _noalloc(L, desc, logits, bias, x, got, stream=None):
    L.moe_route_permute_noalloc(desc, logits, bias, x, got["topk_idx"], got["topk_w"],
                                got["counts"], got["offsets"], got["padded_offsets"],
                                got["tile_prefix"], got["row_src"], got["row_of"], got["x_perm"],
                                stream)


def test_noalloc_route_permute_matches_allocating_call_twice():
    T, E, k, d = 1500, 24, 5, 192
    m, L, desc, logits, bias, x, ref = _routing_case(T, E, k, d)
    for _ in range(2):
        got = _outputs(desc, T, E, k, d, torch.device("cuda"))
        _noalloc(L, desc, logits, bias, x, got)
        torch.cuda.synchronize()
        _compare(got, ref)
    assert m.moe_read_device_status() == 0


def test_noalloc_on_a_side_stream_and_with_no_tokens():
    """The same comparison on a non-default stream, and for a batch with no
    tokens (every count zero, offsets all zero) right after a full one, so
    that nothing the previous call left in the shared array leaks in."""
    T, E, k, d = 700, 16, 3, 128
    m, L, desc, logits, bias, x, ref = _routing_case(T, E, k, d)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    got = _outputs(desc, T, E, k, d, torch.device("cuda"))
    with torch.cuda.stream(side):
        _noalloc(L, desc, logits, bias, x, got, side)
    side.synchronize()
    _compare(got, ref)

    m, L, desc0, logits, bias, x, ref0 = _routing_case(0, E, k, d)
    got0 = _outputs(desc0, 1, E, k, d, torch.device("cuda"))
    _noalloc(L, desc0, logits, bias, x, got0)
    torch.cuda.synchronize()
    assert torch.count_nonzero(got0["counts"]) == 0
    for name in ("counts", "offsets", "padded_offsets", "tile_prefix"):
        assert torch.equal(got0[name], ref0[name]), name
    assert m.moe_read_device_status() == 0


def test_noalloc_rejects_histograms_beyond_the_static_limit():
    import ctypes
    import moe_expert_mlp_gb300 as m

    # ceil(T/256) * E * 4 bytes = 257 * 256 * 4 > 256 KiB
    desc = m.make_desc(T=256 * 257, E=256, k=1, d=64, F=32)
    st = m.lib().moe_route_permute_noalloc(ctypes.byref(desc), *([ctypes.c_void_p(16)] * 12),
                                           ctypes.c_void_p(0))
    assert st == 4          # MOE_ERR_WORKSPACE, nothing enqueued
