"""Pins of the oracle's GLU, expert MLP, combine and analytic backward.

* GLU: closed-form values and torch's own activation routines.
* Forward: a token-by-token MLP written with torch CPU fp64 ops (no grouping,
  no permutation) must equal the oracle's grouped layer.
* Backward: torch autograd of that independent forward, and central finite
  differences of the oracle's own forward on a tiny layer.
* One group of all rows with k=1 is a dense MLP; checked against scalar loops.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle

from tests.test_oracle_route import brute_topk

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------- GLU values
def test_glu_closed_forms():
    P = oracle.GluParams
    one = np.array([1.0])
    zero = np.array([0.0])
    # SiLU: silu(0) = 0, silu'(0) = 1/2, silu(x) -> x for large x
    assert oracle.glu_forward(zero, one, P("swiglu"))[0] == 0.0
    dg, dl = oracle.glu_backward(one, zero, one, P("swiglu"))
    assert dg[0] == 0.5 and dl[0] == 0.0
    assert abs(oracle.glu_forward(np.array([40.0]), one, P("swiglu"))[0] - 40.0) < 1e-12
    # GELU (erf form): gelu(0) = 0, gelu'(0) = 1/2, gelu(x) -> x
    assert oracle.glu_forward(zero, one, P("geglu"))[0] == 0.0
    dg, _ = oracle.glu_backward(one, zero, one, P("geglu"))
    assert abs(dg[0] - 0.5) < 1e-15
    assert abs(oracle.glu_forward(np.array([12.0]), one, P("geglu"))[0] - 12.0) < 1e-12
    # squared ReLU: sReLU(-1) = 0, sReLU(2) = 4, derivative 2*2 = 4
    for act in ("srelu", "sreglu"):
        assert oracle.glu_forward(np.array([-1.0]), one, P(act))[0] == 0.0
        assert oracle.glu_forward(np.array([2.0]), one, P(act))[0] == 4.0
        assert oracle.glu_backward(one, np.array([2.0]), one, P(act))[0][0] == 4.0
    # linear half multiplies; offset adds to it; out_scale scales
    p = P("sreglu", linear_offset=1.0, out_scale=0.5)
    assert oracle.glu_forward(np.array([2.0]), np.array([3.0]), p)[0] == 0.5 * 4.0 * 4.0


def test_glu_clamp_edges():
    p = oracle.GluParams("swiglu", alpha=1.702, limit=7.0, linear_offset=1.0)
    g = np.array([7.0, 7.0 + 1e-9, 9.0, -50.0])
    l = np.array([-7.0, 7.0, 8.0, -1.0])
    a = oracle.glu_forward(g, l, p)
    sig = 1.0 / (1.0 + math.exp(-1.702 * 7.0))
    assert a[0] == pytest.approx(7.0 * sig * (-6.0), rel=1e-14)
    assert a[2] == pytest.approx(7.0 * sig * 8.0, rel=1e-14)        # both clamped
    assert a[3] == pytest.approx(-50.0 / (1.0 + math.exp(1.702 * 50.0)) * 0.0, abs=1e-30)
    dg, dl = oracle.glu_backward(np.ones(4), g, l, p)
    assert dg[0] != 0.0 and dl[0] != 0.0        # bounds included: gradient passes
    assert dg[1] == 0.0 and dl[1] != 0.0        # g just above the limit: stopped
    assert dg[2] == 0.0 and dl[2] == 0.0


@pytest.mark.parametrize("act", ["swiglu", "geglu", "sreglu", "srelu"])
def test_glu_against_torch_routines(act):
    rng = np.random.default_rng(7)
    g = rng.standard_normal(1000) * 4
    l = rng.standard_normal(1000) * 4
    p = oracle.GluParams(act, alpha=1.3 if act == "swiglu" else 1.0, limit=5.0,
                         linear_offset=0.25, out_scale=0.75)
    tg = torch.tensor(g, requires_grad=True)
    tl = torch.tensor(l, requires_grad=True)
    gc = torch.clamp(tg, max=5.0)
    lc = torch.clamp(tl, -5.0, 5.0)
    if act == "swiglu":
        phi = gc * torch.sigmoid(1.3 * gc)
    elif act == "geglu":
        phi = torch.nn.functional.gelu(gc)
    else:
        phi = torch.relu(gc) ** 2
    a = 0.75 * phi * (lc + 0.25) if act != "srelu" else 0.75 * phi
    np.testing.assert_allclose(oracle.glu_forward(g, l, p), a.detach().numpy(), rtol=1e-13, atol=1e-13)
    dA = rng.standard_normal(1000)
    (a * torch.tensor(dA)).sum().backward()
    dg, dl = oracle.glu_backward(dA, g, l, p)
    np.testing.assert_allclose(dg, tg.grad.numpy(), rtol=1e-12, atol=1e-13)
    if act != "srelu":
        np.testing.assert_allclose(dl, tl.grad.numpy(), rtol=1e-12, atol=1e-13)


# ------------------------------------------------------- independent forward
def torch_token_forward(x, logits, bias, W1, b1, W2, b2, k, p):
    """out[t] = sum_s softmax(selected logits)_s * MLP_{e_s}(x[t]), written
    token by token in torch fp64 (selection by brute force)."""
    T, d = x.shape
    E = W1.shape[0]
    F = W2.shape[2]
    score = logits.detach().numpy().astype(np.float32)
    if bias is not None:
        score = score + bias
    outs = []
    for t in range(T):
        sel = brute_topk(list(score[t]), k)
        w = torch.softmax(logits[t, sel].to(torch.float64), dim=0)
        acc = torch.zeros(d, dtype=torch.float64)
        for s, e in enumerate(sel):
            h = W1[e] @ x[t] + (b1[e] if b1 is not None else 0)
            if p.gated:
                g, l = h[:F], h[F:]
            else:
                g, l = h, None
            gc = torch.clamp(g, max=p.limit)
            if p.act == "swiglu":
                phi = gc * torch.sigmoid(p.alpha * gc)
            elif p.act == "geglu":
                phi = torch.nn.functional.gelu(gc)
            else:
                phi = torch.relu(gc) ** 2
            if p.gated:
                a = p.out_scale * phi * (torch.clamp(l, -p.limit, p.limit) + p.linear_offset)
            else:
                a = p.out_scale * phi
            y = W2[e] @ a + (b2[e] if b2 is not None else 0)
            acc = acc + w[s] * y
        outs.append(acc)
    return torch.stack(outs)


def _tiny_layer(seed, T=24, E=5, d=12, F=8, k=2, act="swiglu", bias=True, biases=True):
    rng = np.random.default_rng(seed)
    n1 = 2 * F if act != "srelu" else F
    return dict(
        x=rng.standard_normal((T, d)),
        logits=rng.standard_normal((T, E)).astype(np.float32),
        bias=(rng.standard_normal(E).astype(np.float32) if bias else None),
        W1=rng.standard_normal((E, n1, d)) * 0.3,
        b1=(rng.standard_normal((E, n1)) * 0.1 if biases else None),
        W2=rng.standard_normal((E, d, F)) * 0.3,
        b2=(rng.standard_normal((E, d)) * 0.1 if biases else None),
        dout=rng.standard_normal((T, d)), k=k)


CASES = [
    ("swiglu", dict()),
    ("swiglu", dict(alpha=1.702, limit=1.5, linear_offset=1.0)),
    ("geglu", dict(out_scale=0.5)),
    ("sreglu", dict()),
    ("srelu", dict()),
]


@pytest.mark.parametrize("act,kw", CASES)
def test_forward_and_backward_against_autograd(act, kw):
    L = _tiny_layer(11, act=act)
    p = oracle.GluParams(act, **kw)
    fwd = oracle.moe_forward(L["x"], L["logits"], L["bias"], L["W1"], L["b1"], L["W2"],
                             L["b2"], L["k"], p, align=8)
    bwd = oracle.moe_backward(fwd, L["dout"], L["W1"], L["W2"], p)

    tx = torch.tensor(L["x"], requires_grad=True)
    tlog = torch.tensor(L["logits"].astype(np.float64), requires_grad=True)
    tW1 = torch.tensor(L["W1"], requires_grad=True)
    tb1 = torch.tensor(L["b1"], requires_grad=True)
    tW2 = torch.tensor(L["W2"], requires_grad=True)
    tb2 = torch.tensor(L["b2"], requires_grad=True)
    out = torch_token_forward(tx, tlog, L["bias"], tW1, tb1, tW2, tb2, L["k"], p)
    np.testing.assert_allclose(fwd["out"], out.detach().numpy(), rtol=1e-12, atol=1e-12)
    (out * torch.tensor(L["dout"])).sum().backward()
    for name, got, ref in [("dx", bwd["dx"], tx.grad), ("dlogits", bwd["dlogits"], tlog.grad),
                           ("dW1", bwd["dW1"], tW1.grad), ("db1", bwd["db1"], tb1.grad),
                           ("dW2", bwd["dW2"], tW2.grad), ("db2", bwd["db2"], tb2.grad)]:
        np.testing.assert_allclose(got, ref.numpy(), rtol=1e-10, atol=1e-11, err_msg=name)


def test_backward_finite_differences():
    """Central differences, h = 1e-6, on T=8, d=8, F=4, E=4, k=2 (inputs drawn
    so that no clamp, kink or top-k gap lies near h)."""
    rng = np.random.default_rng(5)
    T, E, d, F, k = 8, 4, 8, 4, 2
    p = oracle.GluParams("swiglu", alpha=1.702, limit=50.0, linear_offset=1.0)
    x = rng.standard_normal((T, d))
    logits = (rng.permuted(np.tile(np.arange(E, dtype=np.float32), (T, 1)), axis=1)
              + np.float32(0.1) * rng.standard_normal((T, E)).astype(np.float32))
    W1 = rng.standard_normal((E, 2 * F, d)) * 0.3
    b1 = rng.standard_normal((E, 2 * F)) * 0.1
    W2 = rng.standard_normal((E, d, F)) * 0.3
    b2 = rng.standard_normal((E, d)) * 0.1
    dout = rng.standard_normal((T, d))

    def loss(x_, lg_, W1_, b1_, W2_, b2_):
        f = oracle.moe_forward(x_, lg_, None, W1_, b1_, W2_, b2_, k, p, align=4)
        return float(np.sum(f["out"] * dout))

    fwd = oracle.moe_forward(x, logits, None, W1, b1, W2, b2, k, p, align=4)
    bwd = oracle.moe_backward(fwd, dout, W1, W2, p)
    h = 1e-6
    args = dict(x_=x, lg_=logits, W1_=W1, b1_=b1, W2_=W2, b2_=b2)
    grads = dict(x_=bwd["dx"], W1_=bwd["dW1"], b1_=bwd["db1"], W2_=bwd["dW2"], b2_=bwd["db2"])
    for name, g in grads.items():
        base = args[name]
        fd = np.zeros_like(base)
        for idx in itertools.product(*[range(n) for n in base.shape]):
            plus = base.copy(); plus[idx] += h
            minus = base.copy(); minus[idx] -= h
            fd[idx] = (loss(**{**args, name: plus}) - loss(**{**args, name: minus})) / (2 * h)
        err = np.max(np.abs(fd - g)) / max(np.max(np.abs(g)), 1e-30)
        assert err < 1e-6, (name, err)
    # logits: perturb in fp64 would change the fp32 selection input; use
    # the softmax path only (selection is fixed because every gap is >= 0.5)
    def loss_logits(lg64):
        f = oracle.moe_forward(x, lg64.astype(np.float32), None, W1, b1, W2, b2, k, p, align=4)
        sel = f["topk_idx"]
        z = np.take_along_axis(lg64, sel, axis=1)
        w = np.exp(z - z.max(1, keepdims=True)); w /= w.sum(1, keepdims=True)
        out = oracle.combine(f["Y"], f["row_of"], w)
        return float(np.sum(out * dout))
    lg64 = logits.astype(np.float64)
    fd = np.zeros_like(lg64)
    for t in range(T):
        for e in range(E):
            pl = lg64.copy(); pl[t, e] += 1e-6
            mi = lg64.copy(); mi[t, e] -= 1e-6
            fd[t, e] = (loss_logits(pl) - loss_logits(mi)) / 2e-6
    err = np.max(np.abs(fd - bwd["dlogits"])) / np.max(np.abs(bwd["dlogits"]))
    assert err < 1e-6, err


def test_one_group_is_a_dense_mlp():
    """E=1, k=1, weight 1: the grouped layer is a dense MLP; checked against
    scalar loops written straight from the definitions."""
    rng = np.random.default_rng(9)
    T, d, F = 6, 5, 3
    x = rng.standard_normal((T, d))
    W1 = rng.standard_normal((1, 2 * F, d))
    b1 = rng.standard_normal((1, 2 * F))
    W2 = rng.standard_normal((1, d, F))
    b2 = rng.standard_normal((1, d))
    p = oracle.GluParams("swiglu")
    fwd = oracle.moe_forward(x, np.zeros((T, 1), np.float32), None, W1, b1, W2, b2, 1, p, align=4)
    assert np.all(fwd["topk_w"] == 1.0)
    for t in range(T):
        h = [b1[0, j] + sum(x[t, c] * W1[0, j, c] for c in range(d)) for j in range(2 * F)]
        a = [h[f] / (1.0 + math.exp(-h[f])) * h[F + f] for f in range(F)]
        for c in range(d):
            y = b2[0, c] + sum(a[f] * W2[0, c, f] for f in range(F))
            assert abs(fwd["out"][t, c] - y) < 1e-12
    # the padded row layout holds the rows in token order
    assert list(fwd["row_src"][:T]) == list(range(T))
