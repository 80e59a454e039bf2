"""Pins of the fp64 backward oracle (CPU only).

The backward oracle is checked against the forward oracle by central finite
differences of L = sum(d_out * out): along random directions of every input
and weight, and element by element on a sample.  Routing is kept away from
ties (top-k margins far above the perturbation), where the layer is smooth.
Planted mistakes in each backward step must break the agreement.  Special
cases: a single expert with top-1 (the router gets no gradient, because the
softmax over one logit is constant) and routing fixed from outside."""
import numpy as np
import pytest

from grouped_gemm_router_gb300 import inputs
from oracle import moe_backward as bwd
from oracle import moe_oracle as orc

EPS = 1e-5
NAMES = ("x", "Wg", "bias", "W1", "W3", "W2", "Ws1", "Ws3", "Ws2")


def _layer(T=12, D=8, F=6, E=4, k=2, shared=True, seed=3):
    _, L = inputs.make_custom(T, D, F, E, k, shared, seed)
    P = {n: orc.bf16_to_f64(L[n]) for n in ("x", "Wg", "W1", "W3", "W2")}
    if shared:
        P.update({n: orc.bf16_to_f64(L[n]) for n in ("Ws1", "Ws3", "Ws2")})
    rng = np.random.default_rng(seed + 100)
    P["bias"] = rng.normal(0, 0.3, E)
    d_out = rng.normal(0, 1, (T, D))
    return P, d_out, k


def _loss(P, d_out, k):
    return bwd.loss(P["x"], P["Wg"], P["W1"], P["W3"], P["W2"], k, d_out, bias=P["bias"],
                    Ws1=P.get("Ws1"), Ws3=P.get("Ws3"), Ws2=P.get("Ws2"))


def _grads(P, d_out, k):
    g = bwd.moe_ffn_backward(P["x"], P["Wg"], P["W1"], P["W3"], P["W2"], k, d_out, bias=P["bias"],
                             Ws1=P.get("Ws1"), Ws3=P.get("Ws3"), Ws2=P.get("Ws2"))
    key = {"x": "dx", "Wg": "dWg", "bias": "dbias", "W1": "dW1", "W3": "dW3", "W2": "dW2",
           "Ws1": "dWs1", "Ws3": "dWs3", "Ws2": "dWs2"}
    return {n: g[key[n]] for n in NAMES if n in P}


def _directional_errors(P, d_out, k, seed=0):
    """Relative error of <grad, v> against the central difference along v."""
    G = _grads(P, d_out, k)
    rng = np.random.default_rng(seed)
    errs = {}
    for n in G:
        v = rng.normal(0, 1, P[n].shape)
        Pp = dict(P); Pp[n] = P[n] + EPS * v
        Pm = dict(P); Pm[n] = P[n] - EPS * v
        fd = (_loss(Pp, d_out, k) - _loss(Pm, d_out, k)) / (2 * EPS)
        an = float((G[n] * v).sum())
        errs[n] = abs(fd - an) / max(abs(fd), 1e-3)
    return errs


def _routing_margin(P, k):
    logits = orc.router_logits(P["x"], P["Wg"], P["bias"])
    return float(orc.topk_gap(logits, k).min())


@pytest.mark.parametrize("T,D,F,E,k,shared,seed", [
    (12, 8, 6, 4, 2, True, 3),
    (10, 16, 8, 6, 3, False, 5),
    (9, 8, 8, 3, 3, True, 8),        # k = E: softmax over every logit
])
def test_gradients_match_central_differences(T, D, F, E, k, shared, seed):
    P, d_out, k = _layer(T, D, F, E, k, shared, seed)
    assert _routing_margin(P, k) > 1e-3     # no selection changes under the perturbation
    errs = _directional_errors(P, d_out, k)
    assert max(errs.values()) < 1e-6, errs


def test_gradients_elementwise_sample():
    P, d_out, k = _layer()
    G = _grads(P, d_out, k)
    rng = np.random.default_rng(9)
    for n in G:
        for _ in range(4):
            idx = tuple(int(rng.integers(0, s)) for s in P[n].shape)
            Pp = {m: a.copy() for m, a in P.items()}; Pp[n][idx] += EPS
            Pm = {m: a.copy() for m, a in P.items()}; Pm[n][idx] -= EPS
            fd = (_loss(Pp, d_out, k) - _loss(Pm, d_out, k)) / (2 * EPS)
            assert abs(fd - G[n][idx]) <= 1e-7 * max(1.0, abs(fd)), (n, idx, fd, G[n][idx])


def test_silu_derivative():
    z = np.linspace(-30, 30, 601)
    num = (orc.silu(z + 1e-6) - orc.silu(z - 1e-6)) / 2e-6
    assert np.abs(bwd.silu_grad(z) - num).max() < 1e-8
    assert bwd.silu_grad(np.array([0.0]))[0] == 0.5                # sigmoid(0) = 1/2
    assert abs(bwd.silu_grad(np.array([40.0]))[0] - 1.0) < 1e-15   # silu(z) -> z
    assert abs(bwd.silu_grad(np.array([-40.0]))[0]) < 1e-15        # silu(z) -> 0


def test_softmax_backward_is_the_jacobian():
    rng = np.random.default_rng(2)
    l = rng.normal(0, 1, 5)
    wb = rng.normal(0, 1, 5)
    sm = lambda a: np.exp(a - a.max()) / np.exp(a - a.max()).sum()
    J = np.array([(sm(l + 1e-6 * np.eye(5)[i]) - sm(l - 1e-6 * np.eye(5)[i])) / 2e-6 for i in range(5)])
    assert np.allclose(bwd.softmax_backward(sm(l), wb), J @ wb, atol=1e-9)
    # shifting every logit leaves the softmax unchanged: the gradient sums to 0
    assert abs(bwd.softmax_backward(sm(l), wb).sum()) < 1e-15


def test_single_expert_top1_router_gets_no_gradient():
    P, d_out, k = _layer(T=8, D=8, F=8, E=1, k=1, shared=False, seed=4)
    g = bwd.moe_ffn_backward(P["x"], P["Wg"], P["W1"], P["W3"], P["W2"], 1, d_out, bias=P["bias"])
    assert not g["dWg"].any() and not g["dbias"].any()
    errs = _directional_errors(P, d_out, 1)
    assert max(errs.values()) < 1e-6, errs


def test_fixed_routing_leaves_router_untouched_and_matches_fd():
    P, d_out, k = _layer(seed=11)
    ids, w = orc.topk_softmax(orc.router_logits(P["x"], P["Wg"], P["bias"]), k)
    g = bwd.moe_ffn_backward(P["x"], P["Wg"], P["W1"], P["W3"], P["W2"], k, d_out, bias=P["bias"],
                             Ws1=P["Ws1"], Ws3=P["Ws3"], Ws2=P["Ws2"], ids=ids, weights=w)
    assert not g["dWg"].any()
    full = _grads(P, d_out, k)
    for n in ("W1", "W3", "W2", "Ws1", "Ws3", "Ws2"):
        assert np.allclose(g["d" + n], full[n], rtol=0, atol=1e-13)
    # dx differs from the routed-through-router one exactly by the router term
    gall = bwd.moe_ffn_backward(P["x"], P["Wg"], P["W1"], P["W3"], P["W2"], k, d_out, bias=P["bias"],
                                Ws1=P["Ws1"], Ws3=P["Ws3"], Ws2=P["Ws2"], return_all=True)
    assert np.allclose(full["x"] - g["dx"], gall["logits_bar"] @ P["Wg"].T, atol=1e-12)


def _swap(mp):
    f = bwd.swiglu_backward
    mp.setattr(bwd, "swiglu_backward", lambda g, u, hb: f(g, u, hb)[::-1])


BACKWARD_MUTATIONS = {
    "silu_grad_is_sigmoid": lambda mp: mp.setattr(bwd, "silu_grad", bwd.sigmoid),
    "g_bar_u_bar_swapped": _swap,
    "softmax_backward_identity": lambda mp: mp.setattr(bwd, "softmax_backward", lambda w, wb: wb),
    "softmax_backward_sign": lambda mp: mp.setattr(
        bwd, "softmax_backward", lambda w, wb: -w * (wb - (w * wb).sum(axis=-1, keepdims=True))),
    "router_gradient_dropped": lambda mp: mp.setattr(bwd, "softmax_backward", lambda w, wb: 0 * wb),
}


@pytest.mark.parametrize("name", sorted(BACKWARD_MUTATIONS))
def test_planted_backward_mistakes_are_caught(name, monkeypatch):
    P, d_out, k = _layer()
    assert max(_directional_errors(P, d_out, k).values()) < 1e-6
    BACKWARD_MUTATIONS[name](monkeypatch)
    assert max(_directional_errors(P, d_out, k).values()) > 1e-3
