"""NVFP4 path against the oracle, through the C-ABI.

* The amax and quantize kernels are checked bit for bit (E2M1 codes, UE4M3
  scale codes, amax values) against the oracle on identical inputs; the
  rotated transposed copy on inputs whose 16-row Hadamard sums are exact in
  fp32 (integers times 2^-6), so both sides decide on the same values.
  Signed zeros compare as zero.
* Each grouped GEMM is checked against the fp64 product of its operands as
  the GPU encoded them (decoded with the oracle's NVFP4 formula), with the
  bf16 bound: this isolates the block-scaled MMA, the scale layout, the
  per-tensor factor 1/(g_a g_b), ragged K tails and the epilogues.
* The whole expert MLP is checked against the NVFP4 oracle
  (grouped_forward_nv / grouped_backward_nv).  H and dH see identically
  quantized operands (bf16 bound); outputs downstream of a requantized
  intermediate (A, dH, or a rotated copy) may see single codes flip where
  accumulation rounding moved a value across a decision boundary, so they
  get max|gpu-ref| <= 0.1 max|ref| and a 2% Frobenius bound.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_mlp_gb300 import _lib as L
from tests import harness as H
from workloads import WORKLOADS, bf16_bits_to_f64, f32_to_bf16_bits, make_inputs, scaled

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]


def _zero_signs(codes):
    codes = np.asarray(codes, dtype=np.uint8)
    return np.where((codes & 7) == 0, 0, codes)


def _inputs(kind, rows, cols, seed):
    rng = np.random.default_rng(seed)
    if kind == "grid":
        v = rng.integers(-127, 128, (rows, cols)).astype(np.float32) * np.float32(2.0 ** -6)
        v[rng.random((rows, cols)) < 0.05] = 0.0
    else:
        v = (rng.standard_normal((rows, cols)) *
             np.exp(rng.standard_normal((rows, 1)))).astype(np.float32)
    bits = f32_to_bf16_bits(v)
    return bits, bf16_bits_to_f64(bits)


def _quantize_gpu(bits, rows, cols, rotate):
    x = H.bits_to_dev(bits)
    amax = torch.zeros(2, dtype=torch.float32, device="cuda")
    L.moe_amax_nvfp4(x, 1, rows, cols, amax)
    u8 = torch.uint8
    out = dict(q=torch.zeros((rows, cols // 2), dtype=u8, device="cuda"),
               scale=torch.zeros(L.moe_nvfp4_scale_bytes(rows, cols), dtype=u8, device="cuda"),
               qt=torch.zeros((cols, rows // 2), dtype=u8, device="cuda"),
               scale_t=torch.zeros(L.moe_nvfp4_scale_bytes(cols, rows), dtype=u8, device="cuda"),
               amax=amax, layout="mma")
    L.moe_quantize_nvfp4_bf16(x, 1, rows, cols, out, rotate_t=rotate)
    torch.cuda.synchronize()
    return {k: (H.to_np(v) if isinstance(v, torch.Tensor) else v) for k, v in out.items()}


def _check_codes(name, q_gpu, sc_gpu_buf, rows, cols, vals, g):
    q_ref, sc_ref, _ = oracle.nvfp4_quantize_rows(vals.astype(np.float32), g)
    codes = H.unpack_fp4_codes(q_gpu)
    assert np.array_equal(_zero_signs(codes), _zero_signs(oracle.e2m1_encode(q_ref))), name
    assert np.array_equal(H.nv_scales_to_rowmajor(sc_gpu_buf, rows, cols), sc_ref), name


@pytest.mark.parametrize("kind,rows,cols", [("grid", 256, 320), ("grid", 96, 128),
                                             ("random", 256, 320), ("random", 384, 192)])
def test_quantizer_bit_exact(kind, rows, cols):
    bits, v = _inputs(kind, rows, cols, seed=rows + cols)
    rotate = kind == "grid"
    out = _quantize_gpu(bits, rows, cols, rotate)
    amax = out["amax"]
    assert amax[0] == np.float32(np.max(np.abs(v)))
    vt = oracle.rht16_rows(v) if rotate else v
    if rotate:                                       # exact sums on the grid inputs
        assert amax[1] == np.float32(np.max(np.abs(vt)))
    _check_codes("rowwise", out["q"], out["scale"], rows, cols, v,
                 oracle.nvfp4_global_scale(amax[0]))
    _check_codes("transposed", out["qt"], out["scale_t"], cols, rows, vt.T,
                 oracle.nvfp4_global_scale(amax[1]))


def test_quantizer_plain_transpose_random():
    """The transposed copy without rotation, on non-grid values, encoded
    with the tensor's amax: bit exact."""
    rows, cols = 192, 256
    bits, v = _inputs("random", rows, cols, seed=5)
    x = H.bits_to_dev(bits)
    a = float(np.max(np.abs(v)))
    amax = torch.tensor([a, a], dtype=torch.float32, device="cuda")
    u8 = torch.uint8
    out = dict(qt=torch.zeros((cols, rows // 2), dtype=u8, device="cuda"),
               scale_t=torch.zeros(L.moe_nvfp4_scale_bytes(cols, rows), dtype=u8, device="cuda"),
               amax=amax, layout="mma")
    L.moe_quantize_nvfp4_bf16(x, 1, rows, cols, out, rotate_t=False)
    torch.cuda.synchronize()
    _check_codes("transposed", H.to_np(out["qt"]), H.to_np(out["scale_t"]), cols, rows, v.T,
                 oracle.nvfp4_global_scale(a))


BASE = WORKLOADS["dsv3_r16384_e32"]
CASES = {
    # K tails: d = 320 is one full K stage plus one MMA; F = 192 three MMAs
    "swiglu_d320": scaled(BASE, R=577, E=4, d=320, F=192, zipf_empty=1, w_std=0.05),
    "gptoss_like": scaled(WORKLOADS["gptoss_t16384_e32"], router="direct", R=450, E=5, d=192,
                          F=192, zipf_s=1.1, zipf_empty=1, w_std=0.05),
    "srelu_nongated": scaled(BASE, R=300, E=3, d=256, F=128, act="srelu", zipf_empty=0,
                             w_std=0.05),
}


def _groups(layer):
    po = H.to_np(layer.padded_offsets)
    cnt = H.to_np(layer.counts)
    return [(e, int(po[e]), int(cnt[e])) for e in range(layer.E) if cnt[e] > 0]


@pytest.mark.parametrize("name", list(CASES))
def test_gemms_on_gpu_codes(name):
    """Every NVFP4 GEMM equals the fp64 product of its GPU-encoded operands."""
    wl = CASES[name]
    inp = make_inputs(wl)
    layer, _ = H.run_both_direct_nv(wl, inp)
    from moe_expert_mlp_gb300 import moe_read_device_status
    assert moe_read_device_status() == 0
    p = H.glu_params(wl)
    E, d, F, W1, cap = layer.E, layer.d, layer.F, layer.W1, layer.capacity
    g = {n: H.to_np(t) for n, t in layer.w_nv.items()}
    wa = g["amax"]
    w1q = [H.nv_dequant(g["w1"][e], g["w1_s"].reshape(E, -1)[e], wa[0], W1, d) for e in range(E)]
    w1tq = [H.nv_dequant(g["w1t"][e], g["w1t_s"].reshape(E, -1)[e], wa[0], d, W1) for e in range(E)]
    w2q = [H.nv_dequant(g["w2"][e], g["w2_s"].reshape(E, -1)[e], wa[2], d, F) for e in range(E)]
    w2tq = [H.nv_dequant(g["w2t"][e], g["w2t_s"].reshape(E, -1)[e], wa[2], F, d) for e in range(E)]

    def act(nv, width, rowwise=True):
        t = {k: H.to_np(v) for k, v in nv.items() if isinstance(v, torch.Tensor)}
        if rowwise:
            return H.nv_dequant(t["q"], t["scale"], t["amax"][0], cap, width)
        return H.nv_dequant(t["qt"], t["scale_t"], t["amax"][1], width, cap)

    Xq, Aq, dYq, dHq = act(layer.x_nv, d), act(layer.a_nv, F), act(layer.dy_nv, d), act(layer.dh_nv, W1)
    Xt, At, dYt, dHt = (act(layer.x_nv, d, False), act(layer.a_nv, F, False),
                        act(layer.dy_nv, d, False), act(layer.dh_nv, W1, False))
    h, a, y = H.to_np(layer.h), H.to_np(layer.a), H.to_np(layer.y)
    dh, dx = H.to_np(layer.dh), H.to_np(layer.dx_perm)
    dw1p, dw2 = H.to_np(layer.dw1p), H.to_np(layer.dw2)
    b1p = H.to_np(layer.b1p) if layer.b1p is not None else None
    b2 = H.to_np(layer.b2) if layer.b2 is not None else None
    got = {k: [] for k in ("H", "Y", "dH", "dX", "dW1", "dW2")}
    ref = {k: [] for k in got}
    for e, lo, m in _groups(layer):
        rows = slice(lo, lo + m)
        hr = Xq[rows] @ w1q[e].T + (b1p[e] if b1p is not None else 0)
        got["H"].append(h[rows]); ref["H"].append(hr)
        yr = Aq[rows] @ w2q[e].T + (b2[e] if b2 is not None else 0)
        got["Y"].append(y[rows]); ref["Y"].append(yr)
        da = dYq[rows] @ w2tq[e].T                        # [m, F]
        hl = H.packed_to_logical_cols(h[rows], F)[0]
        if p.gated:
            dg, dl = oracle.glu_backward(da, hl[:, :F], hl[:, F:], p)
            dhr = np.concatenate([dg, dl], axis=1)
        else:
            dhr = oracle.glu_backward(da, hl, None, p)[0]
        got["dH"].append(H.packed_to_logical_cols(dh[rows], F)[0]); ref["dH"].append(dhr)
        got["dX"].append(dx[rows]); ref["dX"].append(dHq[rows] @ w1tq[e].T)
        k_rows = slice(lo, lo + (m + 63) // 64 * 64)          # K runs to the 64-row step
        got["dW2"].append(dw2[e]); ref["dW2"].append(dYt[:, k_rows] @ At[:, k_rows].T)
        got["dW1"].append(dw1p[e]); ref["dW1"].append(dHt[:, k_rows] @ Xt[:, k_rows].T)
    for k in got:
        H.assert_close(f"{name}/{k}", np.concatenate([x.ravel() for x in got[k]]),
                       np.concatenate([x.ravel() for x in ref[k]]))
    # A = GLU(H) in the FC1 epilogue, and the encode amax values it emits
    for e, lo, m in _groups(layer):
        hl = H.packed_to_logical_cols(h[lo:lo + m], F)[0]
        ar = oracle.glu_forward(hl[:, :F], hl[:, F:], p) if p.gated else oracle.glu_forward(hl, None, p)
        H.assert_close(f"{name}/A", a[lo:lo + m], ar)
    amax_a = H.to_np(layer.a_nv["amax"])
    assert amax_a[0] == np.float32(np.max(np.abs(a)))
    # the requantized A matches the oracle quantizer on the GPU's A, bit for bit
    q_ref, sc_ref, _ = oracle.nvfp4_quantize_rows(
        a[:int(H.to_np(layer.padded_offsets)[-1])].astype(np.float32),
        oracle.nvfp4_global_scale(amax_a[0]))
    R = q_ref.shape[0]
    codes = H.unpack_fp4_codes(H.to_np(layer.a_nv["q"]))[:R]
    assert np.array_equal(_zero_signs(codes), _zero_signs(oracle.e2m1_encode(q_ref)))


@pytest.mark.parametrize("name", list(CASES))
def test_mlp_vs_nvfp4_oracle(name):
    wl = CASES[name]
    inp = make_inputs(wl)
    layer, ref = H.run_both_direct_nv(wl, inp)
    F = wl.F
    got = dict(H=H.packed_to_logical_cols(H.to_np(layer.h), F)[0], A=H.to_np(layer.a),
               Y=H.to_np(layer.y), dH=H.packed_to_logical_cols(H.to_np(layer.dh), F)[0],
               dX_perm=H.to_np(layer.dx_perm),
               dW1=H.to_np(layer.unpack_fc1(layer.dw1p, wl.d)), dW2=H.to_np(layer.dw2))
    if wl.has_b1:
        got["db1"] = H.to_np(layer.unpack_fc1(layer.db1p.reshape(wl.E, -1, 1).contiguous(), 1))[..., 0]
    if wl.has_b2:
        got["db2"] = H.to_np(layer.db2)
    R = int(ref["padded_offsets"][-1])
    for k, g_ in got.items():
        r = ref[k][:R] if k in ("H", "A", "Y", "dH", "dX_perm") else ref[k]
        g_ = g_[:R] if k in ("H", "A", "Y", "dH", "dX_perm") else g_
        if k in ("H", "A", "db2"):
            H.assert_close(f"{name}/{k}", g_, r)
        else:
            H.assert_close(f"{name}/{k}", g_, r, rel=H.TOL_NV, abs_=0.0)
            fro = np.linalg.norm(g_ - r) / max(np.linalg.norm(r), 1e-30)
            assert fro <= H.TOL_NV_FRO, (name, k, fro)


ROUTED = {
    "gptoss_routed": scaled(WORKLOADS["gptoss_t16384_e32"], T=256, E=8, k=4, d=192, F=128,
                            w_std=0.05),
    "max_e256_k32": scaled(WORKLOADS["bf16_t4096_e64"], T=48, E=256, k=32, d=128, F=64,
                           w_std=0.05),
}


def _nv_close(name, got, ref):
    H.assert_close(name, got, ref, rel=H.TOL_NV, abs_=0.0)
    fro = np.linalg.norm(np.asarray(got) - ref) / max(np.linalg.norm(ref), 1e-30)
    assert fro <= H.TOL_NV_FRO, (name, fro)


@pytest.mark.parametrize("name", list(ROUTED))
def test_routed_layer_nvfp4(name):
    """The whole routed step (routing, permute, NVFP4 expert MLP, combine and
    every backward) against the oracle with the NVFP4 expert MLP."""
    wl = ROUTED[name]
    inp = make_inputs(wl)
    ref = H.run_oracle_routed_nv(wl, inp)
    layer = H.run_gpu_routed(wl, inp, layer=H.make_layer(wl, dtype="nvfp4"))
    from moe_expert_mlp_gb300 import moe_read_device_status
    assert moe_read_device_status() == 0
    T = wl.T
    R_pad = int(ref["padded_offsets"][-1])
    assert np.array_equal(H.to_np(layer.topk_idx)[:T], ref["topk_idx"])
    assert np.array_equal(H.to_np(layer.padded_offsets), ref["padded_offsets"])
    H.assert_close("H", H.packed_to_logical_cols(H.to_np(layer.h)[:R_pad], wl.F)[0], ref["H"])
    H.assert_close("A", H.to_np(layer.a)[:R_pad], ref["A"])
    _nv_close("Y", H.to_np(layer.y)[:R_pad], ref["Y"])
    _nv_close("out", H.to_np(layer.out)[:T], ref["out"])
    _nv_close("dH", H.packed_to_logical_cols(H.to_np(layer.dh)[:R_pad], wl.F)[0], ref["dH"])
    _nv_close("dX_perm", H.to_np(layer.dx_perm)[:R_pad], ref["dX_perm"])
    _nv_close("dW2", H.to_np(layer.dw2), ref["dW2"])
    _nv_close("dW1", H.to_np(layer.unpack_fc1(layer.dw1p, wl.d)), ref["dW1"])
    if wl.has_b1:
        db1 = H.to_np(layer.unpack_fc1(layer.db1p.reshape(wl.E, -1, 1).contiguous(), 1))[..., 0]
        _nv_close("db1", db1, ref["db1"])
    if wl.has_b2:
        H.assert_close("db2", H.to_np(layer.db2), ref["db2"])
    _nv_close("dx", H.to_np(layer.dx)[:T], ref["dx"])
    _nv_close("dlogits", H.to_np(layer.dlogits)[:T], ref["dlogits"])


def _direct_nv_layer(wl, inp):
    sizes = inp["group_sizes"]
    _, padded, _ = oracle.group_offsets(sizes, align=128)
    layer = H.make_layer(wl, capacity=max(128, int(padded[-1])), dtype="nvfp4")
    H.load_layer_weights(layer, inp)
    layer.set_groups(torch.from_numpy(sizes.astype(np.int32)).cuda())
    R_pad = int(padded[-1])
    layer.x_perm[:R_pad].copy_(H.bits_to_dev(H.padded_rows(inp["x"], sizes, padded, wl.d)))
    layer.dy[:R_pad].copy_(H.bits_to_dev(H.padded_rows(inp["dout"], sizes, padded, wl.d)))
    return layer


def test_composite_calls_match_per_call_path():
    """moe_mlp_fwd_nv / moe_mlp_bwd_nv give, bit for bit, what the layer's
    sequence of single NVFP4 calls gives."""
    wl = CASES["gptoss_like"]
    inp = make_inputs(wl)
    one = _direct_nv_layer(wl, inp)
    one.mlp_forward()
    one.mlp_backward()
    two = _direct_nv_layer(wl, inp)
    L.moe_mlp_fwd_nv(two.desc, two.x_perm, two.x_nv, two.counts, two.padded_offsets, two.w_nv,
                     two.b1p, two.b2, two.h, two.a, two.a_nv, two.y)
    L.moe_mlp_bwd_nv(two.desc, two.dy, two.dy_nv, two.x_nv, two.h, two.a_nv, two.counts,
                     two.padded_offsets, two.w_nv, two.dh, two.dh_nv, two.dx_perm, two.dw1p,
                     two.db1p, two.dw2, two.db2)
    torch.cuda.synchronize()
    for name in ("h", "a", "y", "dh", "dx_perm", "dw1p", "db1p", "dw2", "db2"):
        t1, t2 = getattr(one, name), getattr(two, name)
        assert torch.equal(t1.view(torch.int16), t2.view(torch.int16)), name


def test_nvfp4_activation_recompute_matches_stored_h():
    """NVFP4 forward without keeping H, backward regenerating it from the
    forward's NVFP4 operands: bitwise the stored H and the same gradients."""
    wl = CASES["gptoss_like"]                       # FC1 bias, clamp, offset
    inp = make_inputs(wl)
    ref = _direct_nv_layer(wl, inp)
    ref.mlp_forward()
    ref.mlp_backward()
    sizes = inp["group_sizes"]
    _, padded, _ = oracle.group_offsets(sizes, align=128)
    rec = H.make_layer(wl, capacity=ref.capacity, dtype="nvfp4", recompute_h=True)
    H.load_layer_weights(rec, inp)
    rec.set_groups(torch.from_numpy(sizes.astype(np.int32)).cuda())
    rec.x_perm.copy_(ref.x_perm)
    rec.dy.copy_(ref.dy)
    rec.mlp_forward()
    rec.mlp_backward()
    assert rec.h is None
    h2 = torch.full_like(ref.h, 7.0)
    L.moe_fc1_recompute_h_nv(rec.desc, rec.x_nv, rec.counts, rec.padded_offsets, rec.w_nv,
                             rec.b1p, h2)
    torch.cuda.synchronize()
    from moe_expert_mlp_gb300 import moe_read_device_status
    assert moe_read_device_status() == 0
    R_pad = int(padded[-1])
    assert torch.equal(h2[:R_pad].view(torch.int16), ref.h[:R_pad].view(torch.int16))
    for name in ("a", "y", "dh", "dx_perm", "dw1p", "db1p", "dw2", "db2"):
        assert torch.equal(getattr(ref, name).view(torch.int16),
                           getattr(rec, name).view(torch.int16)), name
