"""MXFP8 codes and scales from the device quantizer (the one the fused
epilogues use) against the oracle, bit for bit, on identical fp32 inputs."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]


def _edge_blocks():
    """Rows of 32 fp32 values built to hit the rounding and scale edges."""
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = np.unique(np.abs(oracle.e4m3_decode(codes)))           # 0 .. 448
    mids = (vals[:-1] + vals[1:]) / 2                              # exact ties
    rows = []
    X = 2.0 ** -8                                                  # amax 1.0 -> X = 2^-8
    for start in range(0, len(mids), 31):
        r = np.zeros(32)
        r[0] = 448.0 * X                                           # pins the block scale
        seg = mids[start:start + 31] * X
        r[1:1 + len(seg)] = seg * np.where(np.arange(len(seg)) % 2, -1, 1)
        rows.append(r)
    r = np.zeros(32); r[0] = 1.0; r[1] = 464.0 * X; r[2] = -480.0 * X; rows.append(r)  # saturation
    rows.append(np.zeros(32))                                                          # zero block
    r = np.zeros(32); r[0] = 1.0; r[1] = -1e-30; r[2] = -0.0; rows.append(r)           # signed zeros
    r = np.full(32, 2.0 ** -140); r[3] = -3 * 2.0 ** -141; rows.append(r)               # fp32 subnormals
    r = np.linspace(-3e38, 3e38, 32); rows.append(r)                                    # near FLT_MAX
    r = np.zeros(32); r[5] = 0.75; r[6] = 0.75 * 2.0 ** -9; rows.append(r)
    return np.stack(rows).astype(np.float32)


def _random_rows(n, seed):
    rng = np.random.default_rng(seed)
    scale = np.exp2(rng.integers(-40, 40, size=(n, 1)))
    return (rng.standard_normal((n, 32)) * scale).astype(np.float32)


def _run(x, colwise):
    from moe_expert_mlp_gb300 import _lib as L
    xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    rows, cols = x.shape
    if colwise:
        q = torch.empty((cols, rows), dtype=torch.uint8, device="cuda")
        s = torch.empty((cols, rows // 32), dtype=torch.uint8, device="cuda")
    else:
        q = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
        s = torch.empty((rows, cols // 32), dtype=torch.uint8, device="cuda")
    L.moe_quantize_mx(xd, colwise, q, s)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


def test_rowwise_bit_exact():
    for x in (_edge_blocks(), np.ascontiguousarray(_random_rows(4000, 0).reshape(1000, 128))):
        q, s = _run(x, colwise=False)
        q_ref, s_ref = oracle.mx_quantize_rows(x)
        assert np.array_equal(s, s_ref)
        bad = np.argwhere(q != q_ref)
        assert bad.size == 0, (bad[:5], q[tuple(bad[0])], q_ref[tuple(bad[0])])


def test_columnwise_transposed_bit_exact():
    edge = _edge_blocks()                                  # each row becomes one column block
    top = np.ascontiguousarray(edge.T)                     # [32, n_edge]
    rnd = _random_rows(top.shape[1] * 3, 1).reshape(3, top.shape[1], 32).transpose(0, 2, 1)
    x = np.ascontiguousarray(np.concatenate([top] + list(rnd), axis=0))   # [128, n_edge]
    q, s = _run(x, colwise=True)
    q_ref, s_ref = oracle.mx_quantize_cols(x)
    assert np.array_equal(s, s_ref)
    assert np.array_equal(q, q_ref)


# ---------------------------------------------------------------- fused epilogues
from tests import harness as H                       # noqa: E402
from workloads import WORKLOADS, make_inputs, scaled  # noqa: E402


def _check_mx(name, x_bf16, mx, padded, counts):
    """Fused outputs vs the oracle quantizer applied to the stored bf16 tensor."""
    R_pad = int(padded[-1])
    x = H.to_np(x_bf16)[:R_pad].astype(np.float32)
    q_ref, s_ref = oracle.mx_quantize_rows(x)
    assert np.array_equal(mx["q"].cpu().numpy()[:R_pad], q_ref), name + " rowwise codes"
    assert np.array_equal(mx["scale"].cpu().numpy()[:R_pad], s_ref), name + " rowwise scales"
    qt_ref, st_ref = oracle.mx_quantize_cols(x)
    assert np.array_equal(mx["qt"].cpu().numpy()[:, :R_pad], qt_ref), name + " columnwise codes"
    assert np.array_equal(mx["scale_t"].cpu().numpy()[:, :R_pad // 32], st_ref), name + " col scales"
    amax = mx["amax"].cpu().numpy()
    real = np.zeros(R_pad, bool)
    for e, m in enumerate(counts):
        real[int(padded[e]):int(padded[e]) + int(m)] = True
    assert amax[0] == oracle.amax_plain(x, real), name + " amax"
    ref_h = oracle.amax_hadamard_t(x, padded, counts)
    assert abs(amax[1] - ref_h) <= 1e-6 * ref_h + 1e-30, (name, amax[1], ref_h)


@pytest.mark.parametrize("kind", ["routed_bias_clamp", "direct_zipf"])
def test_fused_mx_outputs_of_a_y_dh(kind):
    if kind == "routed_bias_clamp":
        wl = scaled(WORKLOADS["gptoss_t16384_e32"], T=300, E=8, k=4, d=192, F=224)
        inp = make_inputs(wl)
        layer = H.make_layer(wl)
        H.load_layer_weights(layer, inp)
        x = H.bits_to_dev(inp["x"])
        logits = torch.from_numpy(inp["logits"]).cuda()
        layer.route(x, logits, None)
        a_mx, y_mx = layer.mx_buffers(wl.F), layer.mx_buffers(wl.d)
        layer.mlp_forward(a_mx=a_mx, y_mx=y_mx)
        from moe_expert_mlp_gb300 import _lib as L
        L.moe_unpermute_combine(layer.desc, layer.y, layer.row_of, layer.topk_w, layer.out)
        L.moe_unpermute_combine_bwd(layer.desc, H.bits_to_dev(inp["dout"]), layer.y, layer.row_of,
                                    layer.topk_w, layer.row_src, layer.padded_offsets, layer.dy,
                                    layer.dw)
    else:
        wl = scaled(WORKLOADS["dsv3_r16384_e32"], R=900, E=9, d=256, F=192, zipf_empty=3)
        inp = make_inputs(wl)
        layer, _ = H.run_both_direct(wl, inp)
        a_mx, y_mx = layer.mx_buffers(wl.F), layer.mx_buffers(wl.d)
        layer.mlp_forward(a_mx=a_mx, y_mx=y_mx)
    dh_mx = layer.mx_buffers(2 * layer.Fp)
    layer.mlp_backward(dh_mx=dh_mx)
    torch.cuda.synchronize()
    padded = H.to_np(layer.padded_offsets)
    counts = H.to_np(layer.counts)
    _check_mx("A", layer.a, a_mx, padded, counts)
    _check_mx("Y", layer.y, y_mx, padded, counts)
    _check_mx("dH", layer.dh, dh_mx, padded, counts)
