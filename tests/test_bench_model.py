"""bench.py's work models on CPU: algorithmic FLOPs and the attainable-
roofline byte model of the default layer, counted by hand."""
import bench
from workloads import WORKLOADS


def test_default_layer_flops_and_bytes():
    wl = WORKLOADS["bf16_t4096_e64"]
    T, E, k, d, F = 4096, 64, 6, 2048, 1408
    R = T * k
    assert wl.flops_fwd_bwd() == 18 * d * F * R                     # 1.276 TFLOP
    w_el = E * (2 * F * d + d * F)
    weights = 2 * w_el * 2 + 2 * w_el                               # two GEMM reads each, dW once
    per_row = 2 * (10 * d + 5 * 2 * F + 3 * F)                       # x_perm, H, A, Y, dY, dH, dX
    tokens = T * 4 * d * 2 + T * E * 4 * 2                           # x, out, dOut, dx; logits
    assert bench.step_bytes(wl, "bf16") == weights + R * per_row + tokens == 5297405952


def test_block_scaled_byte_models_shrink_operand_bytes():
    wl = WORKLOADS["dsv3_r16384_e32"]
    b16, mx, nv = (bench.step_bytes(wl, t) for t in ("bf16", "mxfp8", "nvfp4"))
    assert nv < mx < b16
    # the dW writes (bf16 in every path) are common to the three
    dw = 2 * wl.E * (2 * wl.F * wl.d + wl.d * wl.F)
    assert nv > dw
