"""fp32 tensors with the grouped GEMMs on the TF32 tensor cores (dtype
"fp32", tcgen05 kind::tf32).

- The tiny fp32 layer (T=256, d=256, E=8, F=512, top-2 SwiGLU) and three
  more routed shapes (biases, GeGLU with F not a multiple of 128, the
  non-gated squared ReLU) run forward and backward through the library on
  fp32 inputs and are compared with the fp64 oracle on the same fp32
  values: routing, offsets and the permuted rows bit-exact, every float
  output within the bf16 bound max|gpu-ref| <= 1e-2 max|ref| + 1e-3.
- Each of the six grouped GEMM calls is exact on operands that TF32 holds
  exactly but bf16 does not (values 1 + j/1024 times a sign, against a
  ternary operand in {-1/4, 0, 1/4}): all partial sums are multiples of
  2^-12 far below 2^24 units, so fp32 accumulation is exact and a result
  off by one bit means the tensor core did not see the TF32 operand.
- The combine backward's dY is bit for bit fp32(w * dout).
- moe_mlp_fwd / moe_mlp_bwd with the fp32 dtype (transposes in the
  workspace) give the same bits as the layer's call sequence.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import harness as H
from workloads import WORKLOADS, make_inputs_fp32, scaled

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

BASE = WORKLOADS["bf16_t4096_e64"]
CASES = {
    "tiny_t256_e8": WORKLOADS["tiny_t256_e8"],
    "bias_geglu_raggedF": scaled(BASE, T=300, E=6, k=3, d=192, F=224, act="geglu",
                                 has_b1=True, has_b2=True, b_std=0.05),
    "srelu_bias": scaled(BASE, T=200, E=5, k=2, d=128, F=160, act="srelu", has_b1=True,
                         b_std=0.05, router_bias=False),
    "swiglu_clamp_k1": scaled(WORKLOADS["gptoss_t16384_e32"], T=160, E=3, k=1, d=64, F=96),
}


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _make_layer(wl, **kw):
    from moe_expert_mlp_gb300 import MoEExpertMLP
    return MoEExpertMLP(wl.E, wl.d, wl.F, T=wl.T, k=wl.k, act=wl.act, alpha=wl.alpha,
                        limit=wl.limit, linear_offset=wl.linear_offset, out_scale=wl.out_scale,
                        has_b1=wl.has_b1, has_b2=wl.has_b2, dtype="fp32", **kw)


def _run_routed(wl):
    f = make_inputs_fp32(wl)
    p = H.glu_params(wl)
    W1, W2 = f["w1"].astype(np.float64), f["w2"].astype(np.float64)
    b1 = f["b1"].astype(np.float64) if f["b1"] is not None else None
    b2 = f["b2"].astype(np.float64) if f["b2"] is not None else None
    fwd = oracle.moe_forward(f["x"].astype(np.float64), f["logits"], f["bias"], W1, b1, W2, b2,
                             wl.k, p, align=128)
    bwd = oracle.moe_backward(fwd, f["dout"].astype(np.float64), W1, W2, p)
    layer = _make_layer(wl)
    layer.load_weights(_dev(f["w1"]), _dev(f["b1"]) if wl.has_b1 else None, _dev(f["w2"]),
                       _dev(f["b2"]) if wl.has_b2 else None)
    bias = _dev(f["bias"]) if f["bias"] is not None else None
    layer.step(_dev(f["x"]), _dev(f["logits"]), bias, _dev(f["dout"]))
    torch.cuda.synchronize()
    return f, fwd, bwd, layer


@pytest.mark.parametrize("name", list(CASES))
def test_fp32_layer_on_tf32_matches_oracle(name):
    wl = CASES[name]
    f, fwd, bwd, layer = _run_routed(wl)
    from moe_expert_mlp_gb300 import moe_read_device_status
    assert moe_read_device_status() == 0
    T, R_pad = wl.T, int(fwd["padded_offsets"][-1])
    n = lambda t: t.cpu().numpy()
    assert np.array_equal(n(layer.topk_idx)[:T], fwd["topk_idx"])
    assert np.array_equal(n(layer.counts), fwd["counts"])
    assert np.array_equal(n(layer.padded_offsets), fwd["padded_offsets"])
    assert np.array_equal(n(layer.row_src)[:R_pad], fwd["row_src"])
    assert np.array_equal(n(layer.row_of)[:T], fwd["row_of"])
    # the permuted rows are copies of fp32 input rows: exact
    assert np.array_equal(n(layer.x_perm)[:R_pad].astype(np.float64), fwd["x_perm"])
    h_log, h_pad = H.packed_to_logical_cols(n(layer.h)[:R_pad].astype(np.float64), wl.F)
    assert np.all(h_pad == 0)
    checks = [("H", h_log, fwd["H"]), ("A", n(layer.a)[:R_pad], fwd["A"]),
              ("Y", n(layer.y)[:R_pad], fwd["Y"]), ("out", n(layer.out)[:T], fwd["out"]),
              ("dY", n(layer.dy)[:R_pad], bwd["dY"]), ("dw", n(layer.dw)[:T], bwd["dw"])]
    dh_log, dh_pad = H.packed_to_logical_cols(n(layer.dh)[:R_pad].astype(np.float64), wl.F)
    assert np.all(dh_pad == 0)
    checks += [("dH", dh_log, bwd["dH"]),
               ("dX_perm", n(layer.dx_perm)[:R_pad], bwd["dX_perm"]),
               ("dW2", n(layer.dw2), bwd["dW2"]),
               ("dW1", n(layer.unpack_fc1(layer.dw1p, wl.d)), bwd["dW1"]),
               ("dx", n(layer.dx)[:T], bwd["dx"]), ("dlogits", n(layer.dlogits)[:T], bwd["dlogits"])]
    if wl.has_b1:
        db1 = n(layer.unpack_fc1(layer.db1p.reshape(wl.E, -1, 1).contiguous(), 1))[..., 0]
        checks.append(("db1", db1, bwd["db1"]))
    if wl.has_b2:
        checks.append(("db2", n(layer.db2), bwd["db2"]))
    for nm, got, ref in checks:
        H.assert_close(nm, got, ref)
        scale = float(np.max(np.abs(ref))) if np.size(ref) else 0.0
        if scale > 0:
            err = float(np.max(np.abs(np.asarray(got, dtype=np.float64) - ref)))
            H.TF32_RATIOS.append((f"{name}.{nm}", err / scale))
    # dY[row_of[t,s]] = fp32(w[t,s] * dout[t]): one fp32 multiply, bit for bit
    w = n(layer.topk_w)[:T]
    dy = n(layer.dy)
    for s in range(wl.k):
        want = (w[:, s:s + 1] * f["dout"]).astype(np.float32)
        assert np.array_equal(dy[fwd["row_of"][:, s]], want)


# ---------------------------------------------------------- exact TF32 grid
def _grid(rng, shape):
    """Values s * (1 + j/1024), j in [0, 1024): 11 significant bits, exact
    in TF32 and (for most j) not in bf16."""
    j = rng.integers(0, 1024, size=shape)
    s = rng.choice([-1.0, 1.0], size=shape)
    return s * (1.0 + j / 1024.0)


def _ternary(rng, shape):
    return rng.choice([-0.25, 0.0, 0.25], size=shape)


def _exact(name, got, ref):
    ref32 = ref.astype(np.float32)
    assert np.array_equal(ref32.astype(np.float64), ref), f"{name}: reference not exact in fp32"
    bad = np.flatnonzero(got.ravel() != ref32.ravel())
    assert bad.size == 0, f"{name}: {bad.size} values differ, first {got.ravel()[bad[0]]} vs {ref32.ravel()[bad[0]]}"


def test_tf32_gemms_exact_on_tf32_grid():
    from moe_expert_mlp_gb300 import _lib as L
    rng = np.random.default_rng(7)
    counts = np.array([130, 0, 77, 1], dtype=np.int32)
    E, d, F = len(counts), 128, 96
    wl = scaled(BASE, T=0, E=E, k=1, d=d, F=F, act="sreglu", router_bias=False)
    _, padded, _ = oracle.group_offsets(counts, align=128)
    R_pad = int(padded[-1])
    cap = R_pad + 128
    layer = _make_layer(wl, capacity=cap)
    layer.set_groups(torch.from_numpy(counts).cuda())
    Fp, W1 = layer.Fp, layer.W1
    real = np.zeros(cap, dtype=bool)
    for e in range(E):
        real[padded[e]:padded[e] + counts[e]] = True
    c, po, desc = layer.counts, layer.padded_offsets, layer.desc

    def rows(vals):                      # zero the padding rows
        v = np.zeros((cap,) + vals.shape[1:])
        v[real] = vals[real]
        return v

    # FC1: H = X W1p^T (grid x ternary), per expert
    X = rows(_grid(rng, (cap, d)))
    w1p = _ternary(rng, (E, W1, d))
    layer.x_perm.copy_(_dev(X))
    layer.w1p.copy_(_dev(w1p))
    L.moe_fc1_glu_fwd_tf32(desc, layer.x_perm, c, po, layer.w1p, None, layer.h, layer.a, None)
    # FC2: Y = A W2^T (grid A x ternary W2)
    A = rows(_grid(rng, (cap, F)))
    w2 = _ternary(rng, (E, d, F))
    a_in, w2_in = _dev(A), _dev(w2)
    L.moe_fc2_fwd_tf32(desc, a_in, c, po, w2_in, None, layer.y)
    # FC2 dgrad + dGLU with H = 1 on both halves (gated squared ReLU, gate
    # 1: phi = 1, phi' = 2), so dL = dA and dG = 2 dA exactly
    dY = rows(_grid(rng, (cap, d)))
    w2t = _ternary(rng, (E, F, d))
    h_ones = torch.ones((cap, W1), dtype=torch.float32, device="cuda")
    dy_in, w2t_in = _dev(dY), _dev(w2t)
    L.moe_fc2_dgrad_dglu_tf32(desc, dy_in, h_ones, c, po, w2t_in, layer.dh, layer.dh_t)
    # FC1 dgrad: dX = dH W1p (grid dH x ternary W1p^T)
    dH = rows(_grid(rng, (cap, W1)))
    w1t = _ternary(rng, (E, d, W1))
    dh_in, w1t_in = _dev(dH), _dev(w1t)
    L.moe_fc1_dgrad_tf32(desc, dh_in, c, po, w1t_in, layer.dx_perm)
    # weight gradients over each group's rows: ternary x grid
    P2, Q2 = rows(_ternary(rng, (cap, d))), rows(_grid(rng, (cap, F)))
    L.moe_fc2_wgrad_tf32(desc, _dev(P2.T), _dev(Q2.T), c, po, layer.dw2)
    P1, Q1 = rows(_grid(rng, (cap, W1))), rows(_ternary(rng, (cap, d)))
    L.moe_fc1_wgrad_tf32(desc, _dev(P1.T), _dev(Q1.T), c, po, layer.dw1p)
    torch.cuda.synchronize()
    from moe_expert_mlp_gb300 import moe_read_device_status
    assert moe_read_device_status() == 0

    n = lambda t: t.cpu().numpy()
    Href, Yref, dAref, dXref = (np.zeros((cap, W1)), np.zeros((cap, d)), np.zeros((cap, Fp)),
                                np.zeros((cap, d)))
    dW2ref, dW1ref = np.zeros((E, d, F)), np.zeros((E, W1, d))
    w2t_pad = np.zeros((E, Fp, d))
    w2t_pad[:, :F] = w2t
    for e in range(E):
        sl = slice(int(padded[e]), int(padded[e]) + int(counts[e]))
        Href[sl] = X[sl] @ w1p[e].T
        Yref[sl] = A[sl] @ w2[e].T
        dAref[sl] = dY[sl] @ w2t_pad[e].T
        dXref[sl] = dH[sl] @ w1t[e].T
        dW2ref[e] = P2[sl].T @ Q2[sl]
        dW1ref[e] = P1[sl].T @ Q1[sl]
    _exact("H", n(layer.h)[:R_pad], Href[:R_pad])
    _exact("Y", n(layer.y)[:R_pad], Yref[:R_pad])
    # dH packed: block b holds gate features 128b.. then linear 128b..
    dHref = np.zeros((cap, W1))
    for f0 in range(0, Fp, 128):
        blk = (f0 // 128) * 256
        dHref[:, blk:blk + 128] = 2.0 * dAref[:, f0:f0 + 128]
        dHref[:, blk + 128:blk + 256] = dAref[:, f0:f0 + 128]
    _exact("dH", n(layer.dh)[:R_pad], dHref[:R_pad])
    _exact("dH^T", n(layer.dh_t)[:, :R_pad], dHref[:R_pad].T)
    _exact("dX", n(layer.dx_perm)[:R_pad], dXref[:R_pad])
    _exact("dW2", n(layer.dw2), dW2ref)
    _exact("dW1p", n(layer.dw1p), dW1ref)
    assert torch.count_nonzero(layer.dw2[1]) == 0 and torch.count_nonzero(layer.dw1p[1]) == 0


def test_fp32_composite_calls_match_layer_sequence():
    """moe_mlp_fwd / moe_mlp_bwd on an fp32 descriptor (the backward makes
    its transposed operands in the workspace) == the layer's per-GEMM call
    sequence, bit for bit."""
    from moe_expert_mlp_gb300 import _lib as L
    wl = CASES["bias_geglu_raggedF"]
    _, fwd, _, layer = _run_routed(wl)
    R_pad = int(fwd["padded_offsets"][-1])
    z = lambda t: torch.zeros_like(t)
    h, a, y = z(layer.h), z(layer.a), z(layer.y)
    L.moe_mlp_fwd(layer.desc, layer.x_perm, layer.counts, layer.padded_offsets, layer.w1p,
                  layer.b1p, layer.w2, layer.b2, h, a, y, ws=layer.ws)
    dh, dxp, dw1p, db1p, dw2, db2 = (z(layer.dh), z(layer.dx_perm), z(layer.dw1p),
                                     z(layer.db1p), z(layer.dw2), z(layer.db2))
    L.moe_mlp_bwd(layer.desc, layer.dy, layer.x_perm, layer.h, layer.a, layer.counts,
                  layer.padded_offsets, layer.w1p, layer.w2, dh, dxp, dw1p, db1p, dw2, db2,
                  ws=layer.ws, b1p=layer.b1p)
    torch.cuda.synchronize()
    for nm, got, want in [("h", h, layer.h), ("a", a, layer.a), ("y", y, layer.y),
                          ("dh", dh, layer.dh), ("dx_perm", dxp, layer.dx_perm)]:
        assert torch.equal(got[:R_pad], want[:R_pad]), nm
    for nm, got, want in [("dw1p", dw1p, layer.dw1p), ("db1p", db1p, layer.db1p),
                          ("dw2", dw2, layer.dw2), ("db2", db2, layer.db2)]:
        assert torch.equal(got, want), nm


def test_fp32_no_tokens_and_empty_groups():
    """T = 0 (every group empty): outputs of the padded layout are empty and
    every weight gradient is exactly zero."""
    wl = scaled(CASES["tiny_t256_e8"], T=0)
    layer = _make_layer(wl)
    rng = np.random.default_rng(3)
    layer.load_weights(_dev(rng.standard_normal((wl.E, 2 * wl.F, wl.d)) * 0.02), None,
                       _dev(rng.standard_normal((wl.E, wl.d, wl.F)) * 0.02), None)
    layer.dw1p.fill_(1.0)
    layer.dw2.fill_(1.0)
    x = torch.zeros((1, wl.d), dtype=torch.float32, device="cuda")
    logits = torch.zeros((1, wl.E), dtype=torch.float32, device="cuda")
    layer.step(x, logits, None, x)
    torch.cuda.synchronize()
    assert int(layer.padded_offsets[-1]) == 0
    assert torch.count_nonzero(layer.dw1p) == 0 and torch.count_nonzero(layer.dw2) == 0
