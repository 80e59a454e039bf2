"""Plain fp64 CPU oracle of the backward pass of the MoE SwiGLU FFN layer.

TEST INFRASTRUCTURE.  Only the tests, the package's smoke check and the
benchmark's CPU-baseline / reference arm may import or run this module.  The
CUDA library never calls it and shares no code with it.

It computes the vector-Jacobian product of the forward pass in
`moe_oracle.moe_ffn_forward` for a scalar loss L = sum(d_out * out): given
d_out = dL/d out [T, D] it returns dL/d x and dL/d every weight.  All values
are float64; nothing is rounded to bf16.

Sources (page title, section):
  [P1] "Triton MoE Kernels & Memory Checkpointing" -- Part A, section 8
       ("Autograd contract"): with g = x W1, u = x W3 and h = silu(g) * u, the
       incoming gradient of h splits into a gradient of g (times u and the
       derivative of silu) and a gradient of u (times silu(g)); the gradient of
       x is the sum of the two transposed products and the weight gradients
       are the outer products of x with those two gradients.  The "dual
       kernels" named there are the hand-written form of this backward.
  [P3] "Chinchilla scaling, MoE, and fused Triton kernels" -- section
       "PyTorch MoE implementation": the forward graph (router logits, top-k,
       softmax over the selected logits, dispatch, grouped GEMMs, weighted
       sum) that the chain rule walks back through here.

Readings:
  * Top-k selection is piecewise constant: logits that are not selected get a
    zero gradient, and the selected ones get the gradient of the softmax over
    the selected logits (the plain derivative of the forward definition away
    from ties).
  * silu'(z) = sigmoid(z) * (1 + z * (1 - sigmoid(z))), the derivative of
    z * sigmoid(z).
  * The shared expert is unweighted, so its output gradient is d_out itself.
"""
from __future__ import annotations

import numpy as np

from . import moe_oracle as fwd


def sigmoid(z: np.ndarray) -> np.ndarray:
    """The logistic function 1 / (1 + exp(-z))."""
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def silu_grad(z: np.ndarray) -> np.ndarray:
    """d/dz [z * sigmoid(z)] = sigmoid(z) + z * sigmoid(z) * (1 - sigmoid(z))."""
    s = sigmoid(z)
    return s * (1.0 + z * (1.0 - s))


def swiglu_backward(g: np.ndarray, u: np.ndarray, h_bar: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """For h = silu(g) * u: dL/dg = h_bar * u * silu'(g), dL/du = h_bar * silu(g)
    [P1 section 8]."""
    return h_bar * u * silu_grad(g), h_bar * fwd.silu(g)


def expert_backward(xs: np.ndarray, W1: np.ndarray, W3: np.ndarray, W2: np.ndarray,
                    y_bar: np.ndarray) -> dict:
    """Backward of one SwiGLU expert y = (silu(xs W1) * (xs W3)) W2 over its rows.
    xs [n, D], W1/W3 [D, F], W2 [F, D], y_bar [n, D].  Returns the gradients of
    xs and the three weights, and the intermediates g, u, h, h_bar, g_bar,
    u_bar."""
    g = xs @ W1
    u = xs @ W3
    h = fwd.silu(g) * u
    h_bar = y_bar @ W2.T
    g_bar, u_bar = swiglu_backward(g, u, h_bar)
    return {
        "xs_bar": g_bar @ W1.T + u_bar @ W3.T,
        "W1_bar": xs.T @ g_bar,
        "W3_bar": xs.T @ u_bar,
        "W2_bar": h.T @ y_bar,
        "g": g, "u": u, "h": h, "h_bar": h_bar, "g_bar": g_bar, "u_bar": u_bar,
    }


def softmax_backward(w: np.ndarray, w_bar: np.ndarray) -> np.ndarray:
    """For w = softmax(l) over the last axis: dL/dl = w * (w_bar - sum(w * w_bar))."""
    return w * (w_bar - (w * w_bar).sum(axis=-1, keepdims=True))


def moe_ffn_backward(x, Wg, W1, W3, W2, k, d_out, bias=None, Ws1=None, Ws3=None, Ws2=None,
                     ids=None, weights=None, return_all=False):
    """Gradients of L = sum(d_out * moe_ffn_forward(...)) in float64.

    Arguments as moe_oracle.moe_ffn_forward (bf16 bit patterns or float64),
    plus d_out [T, D].  With ids/weights given (routing fixed from outside) the
    router receives no gradient.  Returns dict(dx, dWg, dbias, dW1, dW3, dW2
    and, with the shared expert, dWs1, dWs3, dWs2); return_all adds the
    per-slot intermediates (y_bar, w_bar, h_bar, g_bar, u_bar, xs_bar in
    sorted order, logits_bar) and the forward's routing."""
    f = lambda a: a if (a is None or a.dtype == np.float64) else fwd.bf16_to_f64(a)
    x, Wg, W1, W3, W2, d_out = f(x), f(Wg), f(W1), f(W3), f(W2), f(d_out)
    T, D = x.shape
    E, _, F = W1.shape
    routed_in = ids is not None
    logits = fwd.router_logits(x, Wg, bias)
    if routed_in:
        ids = np.asarray(ids, dtype=np.int32)
        w = np.asarray(weights, dtype=np.float64)
    else:
        ids, w = fwd.topk_softmax(logits, k)
    pm = fwd.permutation(ids, E)
    perm, inv, off = pm["perm"].astype(np.int64), pm["inv"].astype(np.int64), pm["offsets"]
    xs = fwd.gather_sorted(x, perm, k)
    S = T * k

    # combine: out[t] = sum_j w[t,j] y[inv[t*k+j]] (+ ys[t])
    tok = perm // k                       # token of each sorted row
    jj = perm % k                         # its slot index j
    y_bar = w[tok, jj][:, None] * d_out[tok]
    # the forward y, per expert, to get the gradient of the gate weights
    y = np.zeros((S, D))
    grads = {"dW1": np.zeros_like(W1), "dW3": np.zeros_like(W3), "dW2": np.zeros_like(W2)}
    xs_bar = np.zeros((S, D))
    inter = {n: np.zeros((S, F)) for n in ("h_bar", "g_bar", "u_bar")}
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        if a == b:
            continue
        r = expert_backward(xs[a:b], W1[e], W3[e], W2[e], y_bar[a:b])
        y[a:b] = r["h"] @ W2[e]
        xs_bar[a:b] = r["xs_bar"]
        grads["dW1"][e], grads["dW3"][e], grads["dW2"][e] = r["W1_bar"], r["W3_bar"], r["W2_bar"]
        for n in inter:
            inter[n][a:b] = r[n]
    w_bar = np.einsum("td,tjd->tj", d_out, y[inv].reshape(T, k, D))

    # un-permute the row gradients: every slot of token t adds into dx[t]
    dx = xs_bar[inv].reshape(T, k, D).sum(axis=1)

    # shared expert: unweighted, so its output gradient is d_out
    if Ws1 is not None:
        rs = expert_backward(x, f(Ws1), f(Ws3), f(Ws2), d_out)
        dx = dx + rs["xs_bar"]
        grads["dWs1"], grads["dWs3"], grads["dWs2"] = rs["W1_bar"], rs["W3_bar"], rs["W2_bar"]

    # router: softmax over the selected logits, zero for the others
    logits_bar = np.zeros((T, E))
    if not routed_in:
        np.put_along_axis(logits_bar, ids.astype(np.int64), softmax_backward(w, w_bar), axis=1)
    dx = dx + logits_bar @ Wg.T
    grads["dx"] = dx
    grads["dWg"] = x.T @ logits_bar
    grads["dbias"] = logits_bar.sum(axis=0)
    if not return_all:
        return grads
    grads.update(y_bar=y_bar, w_bar=w_bar, xs_bar=xs_bar, logits_bar=logits_bar, ids=ids, w=w, **inter, **pm)
    return grads


def loss(x, Wg, W1, W3, W2, k, d_out, bias=None, Ws1=None, Ws3=None, Ws2=None) -> float:
    """L = sum(d_out * out): the scalar whose gradients moe_ffn_backward returns."""
    out = fwd.moe_ffn_forward(x, Wg, W1, W3, W2, k, bias=bias, Ws1=Ws1, Ws3=Ws3, Ws2=Ws2)
    d = d_out if d_out.dtype == np.float64 else fwd.bf16_to_f64(d_out)
    return float((d * out).sum())
