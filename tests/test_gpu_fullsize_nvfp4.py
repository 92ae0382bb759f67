"""Full-size NVFP4 parity: the DeepSeek-shaped layer (16384 rows, 32
experts, d=7168, F=2048) through the same layer and kernels bench.py times
with --dtype nvfp4.

The per-tensor encode scales of x_perm, dY and the weights come from the
inputs, so the oracle computes them in full (plain amax exactly, rotated
amax of x_perm within fp32 rounding) and then, row by row, the quantized
codes of sampled x_perm rows (bit for bit), sampled rows of H (FC1 on the
oracle's NVFP4 operands) and of dH (FC2 dgrad on the oracle's NVFP4
operands, dGLU on the oracle's H).  A and dH's own encode scales need the
whole forward, so the GEMMs downstream of them are checked by properties
that hold at any size: the epilogues' amax equal max |A| and max |dH| of the
stored tensors (and their rotated amax within fp32 rounding), and sampled
rows of Y and dX_perm and sampled columns of dW2 / rows of dW1 equal the
fp64 products of their operands as the GPU encoded them.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import harness as H
from tests.test_gpu_fullsize import _run_gpu
from workloads import WORKLOADS, bf16_bits_to_f64, make_inputs

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]


def _amax_bits(bits):
    """max |x| of bf16 bit patterns (magnitudes order like their bits)."""
    m = np.max(np.asarray(bits, np.uint16) & np.uint16(0x7FFF))
    return float(bf16_bits_to_f64(np.array([m], np.uint16))[0])


def _decode_rows(q, scale_buf, amax, rows, cols, sel, c0=0, c1=None):
    """Decode rows `sel`, columns c0..c1 (multiples of 16) of an NVFP4 tensor
    [rows, cols] as the GPU encoded it."""
    c1 = cols if c1 is None else c1
    codes = H.unpack_fp4_codes(np.asarray(q).reshape(rows, cols // 2)[sel, c0 // 2:c1 // 2])
    s = oracle.e4m3_decode(H.nv_scales_to_rowmajor(scale_buf, rows, cols)[sel, c0 // 16:c1 // 16])
    g = oracle.nvfp4_global_scale(float(amax))
    return oracle.nvfp4_dequantize_rows(H.E2M1_SIGNED[codes], s, g)


def _zs(codes):
    codes = np.asarray(codes, np.uint8)
    return np.where((codes & 7) == 0, 0, codes)


def _rows(t, idx):
    """Rows idx of a device tensor, fetched alone."""
    return H.to_np(t[torch.as_tensor(np.asarray(idx), device=t.device)])


def test_full_size_nvfp4_dsv3():
    wl = WORKLOADS["dsv3_r16384_e32"]
    inp = make_inputs(wl)
    layer = _run_gpu(wl, inp, "nvfp4")
    from moe_expert_mlp_gb300 import moe_read_device_status
    assert moe_read_device_status() == 0
    p = H.glu_params(wl)
    E, d, F, W1, cap = wl.E, wl.d, wl.F, layer.W1, layer.capacity
    sizes = inp["group_sizes"]
    padded = H.to_np(layer.padded_offsets)
    _, padded_ref, _ = oracle.group_offsets(sizes, 128)
    assert np.array_equal(padded, padded_ref)
    starts = np.concatenate([[0], np.cumsum(sizes)])
    rng = np.random.default_rng(13)

    # ---- encode scales from the inputs (oracle, full tensors)
    ax, ady = _amax_bits(inp["x"]), _amax_bits(inp["dout"])
    aw1, aw2 = _amax_bits(inp["w1"]), _amax_bits(inp["w2"])
    xa, dya, wa = (H.to_np(layer.x_nv["amax"]), H.to_np(layer.dy_nv["amax"]),
                   H.to_np(layer.w_nv["amax"]))
    assert (xa[0], dya[0], wa[0], wa[2]) == (np.float32(ax), np.float32(ady), np.float32(aw1),
                                              np.float32(aw2))
    x64 = bf16_bits_to_f64(inp["x"])
    ax_rot = oracle.amax_hadamard_t(x64, starts, sizes)
    assert abs(xa[1] - ax_rot) <= 1e-6 * ax_rot
    del x64

    got, ref = {}, {}

    def add(key, g, r):
        got.setdefault(key, []).append(np.asarray(g, np.float64).ravel())
        ref.setdefault(key, []).append(np.asarray(r, np.float64).ravel())

    nz = np.flatnonzero(sizes > 0)
    experts = sorted({int(nz[np.argmin(sizes[nz])]), int(nz[len(nz) // 2])})
    xq_gpu = H.to_np(layer.x_nv["q"])
    xs_gpu = H.to_np(layer.x_nv["scale"])
    for e in experts:
        m, lo = int(sizes[e]), int(padded[e])
        rows = np.unique([0, m - 1, int(rng.integers(0, m)), int(rng.integers(0, m))])
        X = bf16_bits_to_f64(inp["x"][starts[e] + rows])
        dY = bf16_bits_to_f64(inp["dout"][starts[e] + rows])
        # x_perm codes and scales of the sampled rows, bit for bit
        q_ref, sc_ref, _ = oracle.nvfp4_quantize_rows(X.astype(np.float32),
                                                     oracle.nvfp4_global_scale(ax))
        codes = H.unpack_fp4_codes(xq_gpu[lo + rows])
        assert np.array_equal(_zs(codes), _zs(oracle.e2m1_encode(q_ref)))
        assert np.array_equal(H.nv_scales_to_rowmajor(xs_gpu, cap, d)[lo + rows], sc_ref)
        # H and dH rows on the oracle's NVFP4 operands
        W1e = bf16_bits_to_f64(inp["w1"][e])
        W2e = bf16_bits_to_f64(inp["w2"][e])
        Hr = oracle.nvfp4_fake_rows(X, ax) @ oracle.nvfp4_fake_rows(W1e, aw1).T
        add("H", H.packed_to_logical_cols(_rows(layer.h, lo + rows), F)[0], Hr)
        dA = oracle.nvfp4_fake_rows(dY, ady) @ oracle.nvfp4_fake_cols(W2e, aw2)
        H16 = oracle.bf16_round(Hr)
        dg, dl = oracle.glu_backward(dA, H16[:, :F], H16[:, F:], p)
        add("dH", H.packed_to_logical_cols(_rows(layer.dh, lo + rows), F)[0],
            np.concatenate([dg, dl], 1))
    for key in got:
        H.assert_close(f"dsv3_nvfp4/{key}", np.concatenate(got[key]), np.concatenate(ref[key]))

    # ---- properties downstream of A's and dH's own encode scales
    R_pad = int(padded[-1])
    real = np.zeros(R_pad, bool)
    for e in range(E):
        real[int(padded[e]):int(padded[e]) + int(sizes[e])] = True
    a = H.to_np(layer.a)[:R_pad]
    aa, dha = H.to_np(layer.a_nv["amax"]), H.to_np(layer.dh_nv["amax"])
    assert aa[0] == np.float32(np.max(np.abs(a[real])))
    real_t = torch.from_numpy(real).to(layer.dh.device)
    assert dha[0] == np.float32(layer.dh[:R_pad][real_t].float().abs().max().item())
    a_rot = oracle.amax_hadamard_t(a, padded, sizes)
    assert abs(aa[1] - a_rot) <= 1e-6 * a_rot
    g = {n: H.to_np(t) for n, t in layer.w_nv.items()}
    an = {k: H.to_np(v) for k, v in layer.a_nv.items() if isinstance(v, torch.Tensor)}
    dhn = {k: H.to_np(v) for k, v in layer.dh_nv.items() if isinstance(v, torch.Tensor)}
    dyn = {k: H.to_np(v) for k, v in layer.dy_nv.items() if isinstance(v, torch.Tensor)}
    xn = {k: H.to_np(v) for k, v in layer.x_nv.items() if isinstance(v, torch.Tensor)}
    got, ref = {}, {}
    for e in experts:
        m, lo = int(sizes[e]), int(padded[e])
        sel = lo + np.unique([0, m - 1, int(rng.integers(0, m))])
        w2q = H.nv_dequant(g["w2"][e], g["w2_s"].reshape(E, -1)[e], wa[2], d, F)
        w1tq = H.nv_dequant(g["w1t"][e], g["w1t_s"].reshape(E, -1)[e], wa[0], d, W1)
        add("Y", _rows(layer.y, sel), _decode_rows(an["q"], an["scale"], aa[0], cap, F, sel) @ w2q.T)
        add("dX", _rows(layer.dx_perm, sel),
            _decode_rows(dhn["q"], dhn["scale"], dha[0], cap, W1, sel) @ w1tq.T)
        # weight gradients: K over the group's rows up to the next multiple of 64
        k_end = lo + (m + 63) // 64 * 64
        cols = np.unique([0, F - 1, int(rng.integers(0, F))])
        dYt = _decode_rows(dyn["qt"], dyn["scale_t"], dya[1], d, cap, np.arange(d), lo, k_end)
        At = _decode_rows(an["qt"], an["scale_t"], aa[1], F, cap, cols, lo, k_end)
        add("dW2", H.to_np(layer.dw2[e][:, torch.as_tensor(cols, device=layer.dw2.device)]),
            dYt @ At.T)
        prow = np.unique([0, W1 - 1, int(rng.integers(0, W1))])
        dHt = _decode_rows(dhn["qt"], dhn["scale_t"], dha[1], W1, cap, prow, lo, k_end)
        Xt = _decode_rows(xn["qt"], xn["scale_t"], xa[1], d, cap, np.arange(d), lo, k_end)
        add("dW1", _rows(layer.dw1p[e], prow), dHt @ Xt.T)
    for key in got:
        H.assert_close(f"dsv3_nvfp4/{key}", np.concatenate(got[key]), np.concatenate(ref[key]))
