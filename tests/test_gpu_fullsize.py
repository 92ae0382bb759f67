"""Full-size parity: the bench's workloads at their full sizes, run through
the same layer and kernels (same launch configuration) that bench.py times.
The oracle checks the routing in full and, one by one, sampled outputs:
rows of H, A, Y, dH and dX_perm; for routed layers whole tokens of out, dx,
dw and dlogits; and rows of dW1 / columns of dW2, each with the full
reduction over its expert's rows.  Tolerances as in the small parity tests:
max|gpu-ref| <= 1e-2 max|ref| + 1e-3 over the sampled values against the
oracle with the same operand format (bf16, or MXFP8 quantized the same way);
on the MXFP8 path also a relative Frobenius error <= 1e-1 against the
unquantized oracle (the format's own error is 6-8 %).  The fp32 layer (TF32
GEMMs) is held to the bf16 bound against the plain oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import harness as H
from workloads import WORKLOADS, bf16_bits_to_f64, make_inputs

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

CASES = [("bf16_t4096_e64", "bf16"), ("dsv3_r16384_e32", "bf16"), ("dsv3_r16384_e32", "mxfp8"),
         ("gptoss_t16384_e32", "mxfp8"), ("dense_m16384", "bf16"),
         # the fp32 layer (TF32 GEMMs) at the DeepSeek-shaped size, on the same
         # (bf16-valued) inputs held in fp32
         ("dsv3_r16384_e32", "fp32")]


def _run_gpu(wl, inp, dtype):
    """The full layer on the GPU, as bench.py runs it (one eager step)."""
    routed = wl.router != "direct"
    if routed:
        layer = H.make_layer(wl, dtype=dtype)
        H.run_gpu_routed(wl, inp, layer=layer)
        return layer
    sizes = inp["group_sizes"]
    cap = max(128, int(sum((int(m) + 127) // 128 * 128 for m in sizes)))
    layer = H.make_layer(wl, capacity=cap, dtype=dtype)
    f32 = dtype == "fp32"
    dev = (lambda b: H.bits_to_dev(b).float()) if f32 else H.bits_to_dev
    if f32:
        opt = lambda b: dev(b) if b is not None else None
        layer.load_weights(dev(inp["w1"]), opt(inp["b1"]), dev(inp["w2"]), opt(inp["b2"]))
    else:
        H.load_layer_weights(layer, inp)
    layer.set_groups(torch.from_numpy(sizes.astype(np.int32)).cuda())
    po = H.to_np(layer.padded_offsets)
    xs, dys = dev(inp["x"]), dev(inp["dout"])
    src = 0
    for e, m in enumerate(sizes):
        m = int(m)
        layer.x_perm[po[e]:po[e] + m].copy_(xs[src:src + m])
        layer.dy[po[e]:po[e] + m].copy_(dys[src:src + m])
        src += m
    layer.grouped_step()
    torch.cuda.synchronize()
    return layer


class _Expert:
    """One expert's weights in fp64, converted on demand."""

    def __init__(self, inp, e):
        self.W1 = bf16_bits_to_f64(inp["w1"][e])
        self.W2 = bf16_bits_to_f64(inp["w2"][e])
        self.b1 = bf16_bits_to_f64(inp["b1"][e]) if inp["b1"] is not None else None
        self.b2 = bf16_bits_to_f64(inp["b2"][e]) if inp["b2"] is not None else None


def _rows_fwd_bwd(ex, X, dY, p, mx):
    """Row-wise forward and backward of one expert for the given rows (each
    output row depends on its own input row only; the weight-gradient outputs
    of the oracle call are not used here)."""
    if mx:
        Hh, A, Y = oracle.expert_forward_mx(X, ex.W1, ex.b1, ex.W2, ex.b2, p)
        dX, dH = oracle.expert_backward_mx(X, Hh, A, dY, ex.W1, ex.W2, p)[:2]
    else:
        Hh, A, Y = oracle.expert_forward(X, ex.W1, ex.b1, ex.W2, ex.b2, p)
        dX, dH = oracle.expert_backward(X, Hh, A, dY, ex.W1, ex.W2, p)[:2]
    return Hh, A, Y, dX, dH


def _pad32(v):
    out = np.zeros(((v.shape[0] + 31) // 32 * 32,) + v.shape[1:])
    out[:v.shape[0]] = v
    return out


def _dw_samples(ex, Xe, dYe, p, mx, cols):
    """dW2[:, j] and dW1 rows (gate j, linear F+j) for the sampled features,
    each reduced over all rows of the expert."""
    F = ex.W2.shape[1]
    gated = p.gated
    Xr = oracle.mx_fake_rows(Xe) if mx else Xe
    out = {}
    for j in cols:
        rows = [j, F + j] if gated else [j]
        W1r = oracle.mx_fake_rows(ex.W1[rows]) if mx else ex.W1[rows]
        Hc = Xr @ W1r.T
        if ex.b1 is not None:
            Hc = Hc + ex.b1[rows][None, :]
        A = oracle.glu_forward(Hc[:, 0], Hc[:, 1] if gated else None, p)
        if mx:
            A16 = oracle.bf16_round(A)
            H16 = oracle.bf16_round(Hc)
            dYq = oracle.mx_fake_cols(_pad32(dYe))
            dW2c = dYq.T @ oracle.mx_fake_cols(_pad32(A16[:, None]))[:, 0]
            dA = oracle.mx_fake_rows(dYe) @ oracle.mx_fake_cols(ex.W2[:, j:j + 1])[:, 0]
            g = oracle.glu_backward(dA, H16[:, 0], H16[:, 1] if gated else None, p)
            Xc = oracle.mx_fake_cols(_pad32(Xe))
            dW1 = [oracle.mx_fake_cols(_pad32(oracle.bf16_round(gi)[:, None]))[:, 0] @ Xc
                   for gi in g if gi is not None]
        else:
            dW2c = dYe.T @ A
            dA = dYe @ ex.W2[:, j]
            g = oracle.glu_backward(dA, Hc[:, 0], Hc[:, 1] if gated else None, p)
            dW1 = [gi @ Xe for gi in g if gi is not None]
        out[j] = (dW2c, dW1)
    return out


@pytest.mark.parametrize("name,dtype", CASES)
def test_full_size_sampled(name, dtype):
    wl = WORKLOADS[name]
    mx = dtype == "mxfp8"
    inp = make_inputs(wl)
    layer = _run_gpu(wl, inp, dtype)
    from moe_expert_mlp_gb300 import moe_read_device_status
    assert moe_read_device_status() == 0
    p = H.glu_params(wl)
    F, k = wl.F, wl.k
    rng = np.random.default_rng(11)
    got, ref, plain = {}, {}, {}

    def add(key, g, r, r_plain=None):
        got.setdefault(key, []).append(np.asarray(g, np.float64).ravel())
        ref.setdefault(key, []).append(np.asarray(r, np.float64).ravel())
        if r_plain is not None:
            plain.setdefault(key, []).append(np.asarray(r_plain, np.float64).ravel())

    gpu = {n: H.to_np(getattr(layer, n)) for n in ("h", "a", "y", "dh", "dx_perm")}
    h_log = H.packed_to_logical_cols(gpu["h"], F)[0]
    dh_log = H.packed_to_logical_cols(gpu["dh"], F)[0]
    routed = wl.router != "direct"
    if routed:
        # the routing in full, bit for bit
        topk_idx, topk_w, counts = oracle.route(inp["logits"], inp["bias"], k)
        _, padded, _ = oracle.group_offsets(counts, 128)
        row_src, row_of = oracle.permute_index(topk_idx, wl.E, padded)
        assert np.array_equal(H.to_np(layer.topk_idx)[:wl.T], topk_idx)
        assert np.array_equal(H.to_np(layer.counts), counts)
        assert np.array_equal(H.to_np(layer.padded_offsets), padded)
        assert np.array_equal(H.to_np(layer.row_of)[:wl.T], row_of)
        sizes = counts
    else:
        sizes = inp["group_sizes"]
        padded = H.to_np(layer.padded_offsets)
        starts = np.concatenate([[0], np.cumsum(sizes)])
    nz = np.flatnonzero(sizes > 0)
    sample_experts = sorted({int(nz[np.argmin(sizes[nz])]), int(nz[len(nz) // 2])})

    def group_rows(e):
        """All rows of expert e: inputs X and upstream gradients dY (fp64)."""
        m, lo = int(sizes[e]), int(padded[e])
        if not routed:
            return (bf16_bits_to_f64(inp["x"][starts[e]:starts[e] + m]),
                    bf16_bits_to_f64(inp["dout"][starts[e]:starts[e] + m]))
        toks = row_src[lo:lo + m]                       # token of each row
        slot = np.argmax(topk_idx[toks] == e, axis=1)
        dY = topk_w[toks, slot][:, None] * bf16_bits_to_f64(inp["dout"][toks])
        return bf16_bits_to_f64(inp["x"][toks]), (oracle.bf16_round(dY) if mx else dY)

    # sampled rows: (expert, padded row, x row, dY row), evaluated per expert
    rows = []
    for e in sample_experts:
        Xe, dYe = group_rows(e)
        m = Xe.shape[0]
        for r in np.unique([0, m - 1, int(rng.integers(0, m))]):
            rows.append((e, int(padded[e]) + int(r), Xe[r], dYe[r]))
    toks = []
    if routed:                                          # whole tokens (all k slots)
        n_tok = 6
        toks = [int(t) for t in np.unique(np.concatenate([[wl.T - 1], rng.integers(0, wl.T, n_tok - 1)]))]
        for t in toks:
            x = bf16_bits_to_f64(inp["x"][t])
            dout = bf16_bits_to_f64(inp["dout"][t])
            for s_ in range(k):
                dy = float(topk_w[t, s_]) * dout
                rows.append((int(topk_idx[t, s_]), int(row_of[t, s_]), x,
                             oracle.bf16_round(dy) if mx else dy))
    Yrow, dXrow = {}, {}
    for e in sorted({r[0] for r in rows}):
        sel = [r for r in rows if r[0] == e]
        ex = _Expert(inp, e)
        Xs, dYs = np.stack([r[2] for r in sel]), np.stack([r[3] for r in sel])
        Hh, A, Y, dX, dHr = _rows_fwd_bwd(ex, Xs, dYs, p, mx)
        Hu, Au, Yu, dXu, dHu = _rows_fwd_bwd(ex, Xs, dYs, p, False) if mx else [None] * 5
        for i, (_, row, _, _) in enumerate(sel):
            add("H", h_log[row], Hh[i])
            add("A", gpu["a"][row], A[i])
            add("Y", gpu["y"][row], Y[i], Yu[i] if mx else None)
            add("dH", dh_log[row], dHr[i], dHu[i] if mx else None)
            add("dX_perm", gpu["dx_perm"][row], dX[i], dXu[i] if mx else None)
            Yrow[row], dXrow[row] = Y[i], dX[i]
            if mx:
                Yrow[("u", row)], dXrow[("u", row)] = Yu[i], dXu[i]
        if e in sample_experts:                         # weight gradients, full reduction
            Xe, dYe = group_rows(e)
            cols = np.unique([0, F - 1, int(rng.integers(0, F))])
            dw1_gpu = H.to_np(layer.unpack_fc1(layer.dw1p, wl.d))[e]
            dw2_gpu = H.to_np(layer.dw2)[e]
            samples = _dw_samples(ex, Xe, dYe, p, mx, cols)
            samples_u = _dw_samples(ex, Xe, dYe, p, False, cols) if mx else None
            for j, (dW2c, dW1) in samples.items():
                u2, u1 = samples_u[j] if mx else (None, [None, None])
                add("dW2", dw2_gpu[:, j], dW2c, u2)
                add("dW1", dw1_gpu[j], dW1[0], u1[0])
                if p.gated:
                    add("dW1", dw1_gpu[F + j], dW1[1], u1[1])
    if routed:
        dw_gpu, dl_gpu = H.to_np(layer.dw), H.to_np(layer.dlogits)
        for t in toks:
            dout = bf16_bits_to_f64(inp["dout"][t])
            slots = [int(row_of[t, s_]) for s_ in range(k)]
            out_t = sum(float(topk_w[t, s_]) * Yrow[r] for s_, r in enumerate(slots))
            dw_t = np.array([float(np.dot(dout, Yrow[r])) for r in slots])
            dl_t = oracle.route_backward(dw_t[None], topk_w[t][None], topk_idx[t][None], wl.E)[0]
            u = {}
            if mx:
                dw_u = np.array([float(np.dot(dout, Yrow[("u", r)])) for r in slots])
                u = dict(out=sum(float(topk_w[t, s_]) * Yrow[("u", r)]
                                 for s_, r in enumerate(slots)),
                         dx=sum(dXrow[("u", r)] for r in slots), dw=dw_u,
                         dlogits=oracle.route_backward(dw_u[None], topk_w[t][None],
                                                       topk_idx[t][None], wl.E)[0])
            add("out", H.to_np(layer.out)[t], out_t, u.get("out"))
            add("dx", H.to_np(layer.dx)[t], sum(dXrow[r] for r in slots), u.get("dx"))
            add("dw", dw_gpu[t], dw_t, u.get("dw"))
            add("dlogits", dl_gpu[t], dl_t, u.get("dlogits"))
    for key in got:
        g, r = np.concatenate(got[key]), np.concatenate(ref[key])
        if key in ("H", "A") or not mx:                 # H, A: identical operands
            H.assert_close(f"{name}/{dtype}/{key}", g, r)
        else:
            H.assert_mx(f"{name}/{dtype}/{key}", g, r, np.concatenate(plain[key]))
