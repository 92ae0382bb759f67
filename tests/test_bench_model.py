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


def test_fp32_byte_model_of_the_tiny_layer():
    """fp32 tensors (TF32 GEMMs): 4-byte elements, and the weight gradients
    read transposed copies of x_perm, A, dY and dH (x_perm and dY through a
    transpose pass that reads and writes them once)."""
    wl = WORKLOADS["tiny_t256_e8"]
    T, E, k, d, F = 256, 8, 2, 256, 512
    R = T * k
    w_el = E * (2 * F * d + d * F)
    weights = 2 * w_el * 4 + w_el * 4                               # two GEMM reads each, dW once
    per_row = 4 * (5 * d + 2 * 2 * F + 4 * F + 2 * d + 5 * d + 4 * 2 * F + 2 * d)
    tokens = T * 4 * d * 4 + T * E * 4 * 2
    assert bench.step_bytes(wl, "fp32") == weights + R * per_row + tokens
    assert bench.call_work(wl, "transpose_x", R, "fp32") == ("byte", R * d * 8.0)
    assert bench.call_work(wl, "combine", R, "fp32") == ("byte", 2.0 * (R * d * 2 + T * d * 2))
    assert bench.call_work(wl, "fc1_glu_fwd", R, "fp32") == ("flop", 2.0 * R * d * 2 * F)


def test_weight_gradient_bytes_pick_the_hbm_roof_on_mxfp8():
    """FC1 weight gradient of the DeepSeek-shaped layer: the transposed
    MXFP8 copies of dH and x_perm read once (a scale per 32 codes) and dW1
    written once in bf16 -- 2.07 GB, which at the measured 6789 GB/s takes
    longer than its 0.962 TFLOP at twice the measured bf16 peak, so the HBM
    roof bounds it; in bf16 the tensor roof does."""
    wl = WORKLOADS["dsv3_r16384_e32"]
    R, E, d, F = 16384, 32, 7168, 2048
    q = 1 + 1 / 32
    want = R * 2 * F * q + R * d * q + E * 2 * F * d * 2
    assert bench.gemm_bytes(wl, "fc1_wgrad", R, "mxfp8") == want
    flops = bench.call_work(wl, "fc1_wgrad", R, "mxfp8")[1]
    assert want / 6789.3e9 > flops / (2 * 1889.5e12)
    b16 = bench.gemm_bytes(wl, "fc1_wgrad", R, "bf16")
    assert b16 == R * 2 * F * 2 + R * d * 2 + E * 2 * F * d * 2
    assert b16 / 6789.3e9 < flops / 1889.5e12
