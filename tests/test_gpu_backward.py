"""Parity of the backward pass (moe_ffn_backward, through the C ABI) with the
fp64 backward oracle.

Tolerances.  The GPU stores y_bar, h_bar, g_bar | u_bar, h and x_bar as bf16
between its GEMMs (relative rounding 2^-9 each) and accumulates in fp32:
  * dx sums the k + 1 slot gradients of a token, each a 2F-long contraction
    of bf16-rounded g_bar / u_bar (which carry the roundings of y_bar and
    h_bar before them): its error is ~2^-8 rms(dx), so
    |gpu - oracle| <= 2.5e-2 rms(oracle) + 1e-2 |oracle| (about six standard
    deviations);
  * weight gradients (sums over an expert's rows of products whose factors
    carry up to ~2^-7 relative rounding from the bf16 intermediates, with
    independent signs): the error of an entry is ~2^-7 rms(oracle), so
    |gpu - oracle| <= 5e-2 rms(oracle) + 1e-2 |oracle| per tensor (about six
    standard deviations, for tensors of ~10^5 entries).
Stage checks feed the oracle the GPU's own bf16 intermediates (read from
the backward workspace), so each GEMM is held to its fp32 accumulation:
h_bar, x_bar: 1e-4 + 4e-3 |ref|; g_bar | u_bar: 2e-3 rms + 8e-3 |ref|; weight
gradients: 1e-3 rms + 1e-3 |ref|; and the h the backward recomputes after a
chained forward equals the unchained forward's h bit for bit (same kernel
arithmetic).
Routing: the small cases use seeds whose top-k margins all exceed 1e-3 (the
router's selection is then the oracle's, and the router gradients are
compared); the full-size case fixes the routing from outside (no router
gradient) and checks sampled columns of every gradient."""
import numpy as np
import pytest
import torch

from grouped_gemm_router_gb300 import inputs
from oracle import moe_backward as bwd
from oracle import moe_oracle as orc

from _util import assert_close, to_dev, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from grouped_gemm_router_gb300 import build
    build.build()
    from grouped_gemm_router_gb300 import moe as m
    return m


H_RTOL, H_ATOL = 4e-3, 1e-4


def _rms(a):
    return max(float(np.sqrt(np.mean(a ** 2))) if a.size else 0.0, 1e-6)


def assert_wgrad(got, ref, what, scale=5e-2, rtol=1e-2):
    assert_close(got, ref, what, atol=scale * _rms(ref), rtol=rtol)


def assert_dx(got, ref, what="dx"):
    assert_close(got, ref, what, atol=2.5e-2 * _rms(ref), rtol=1e-2)


def _d_out(T, D, seed):
    rng = np.random.default_rng(seed)
    return inputs.f32_to_bf16_bits(rng.standard_normal((T, D)).astype(np.float32))


def _run(moe, L, k, d_out_bits, shared, chained=False, ids_in=None, weights_in=None, router=True):
    G = {key: (to_dev(v) if v is not None else None) for key, v in L.items()}
    T, D = L["x"].shape
    E, _, F = L["W1"].shape
    ws = moe.Workspace(T, D, F, E, k, shared)
    bws = moe.BackwardWorkspace(T, D, F, E, k, shared)
    kw = dict(Ws1=G["Ws1"], Ws3=G["Ws3"], Ws2=G["Ws2"]) if shared else {}
    out = moe.moe_ffn_forward(G["x"], G["Wg"], G["W1"], G["W3"], G["W2"], k, bias=G["bias"], workspace=ws,
                              ids_in=ids_in, weights_in=weights_in, chained=chained, **kw)
    g = moe.moe_ffn_backward(G["x"], G["Wg"], G["W1"], G["W3"], G["W2"], k, to_dev(d_out_bits), ws,
                             bwd_workspace=bws, ids_in=ids_in, weights_in=weights_in, router=router,
                             chained=chained, **kw)
    torch.cuda.synchronize()
    assert moe.device_error() == 0
    return out, g, (ws, bws)


def _stage_checks(moe, L, k, d_out, g, wss, shared):
    """Each backward GEMM against the oracle applied to the GPU's own bf16
    inputs, in sorted order."""
    ws, bws = wss
    V, B = ws.views(), bws.views()
    T, D = L["x"].shape
    E, _, F = L["W1"].shape
    S = T * k
    counts = V["counts"].cpu().numpy()
    offs = V["offsets"].cpu().numpy()
    prow = torch.tensor(moe.padded_rows(counts), dtype=torch.long, device="cuda")
    Sp = B["S_pad"]
    W1, W3, W2 = (orc.bf16_to_f64(L[n]) for n in ("W1", "W3", "W2"))
    xs = to_f64(V["x_sorted"])
    ybar, hbar = to_f64(B["ybar"][prow]), to_f64(B["hbar"][prow])
    gu, xbar = to_f64(B["gu"][prow]), to_f64(B["xbar"][prow])
    hbw = V["h"][:S]  # the W2 gradient reads the forward's h
    for e in range(E):
        a, b = int(offs[e]), int(offs[e + 1])
        if a == b:
            continue
        assert_close(hbar[a:b], ybar[a:b] @ W2[e].T, f"h_bar e{e}", atol=H_ATOL, rtol=H_RTOL)
        gref, uref = bwd.swiglu_backward(xs[a:b] @ W1[e], xs[a:b] @ W3[e], hbar[a:b])
        assert_close(gu[a:b, :F], gref, f"g_bar e{e}", atol=2e-3 * _rms(gref), rtol=8e-3)
        assert_close(gu[a:b, F:], uref, f"u_bar e{e}", atol=2e-3 * _rms(uref), rtol=8e-3)
        assert_close(xbar[a:b], gu[a:b, :F] @ W1[e].T + gu[a:b, F:] @ W3[e].T, f"x_bar e{e}",
                     atol=H_ATOL, rtol=H_RTOL)
        assert_wgrad(to_f64(g["dW1"][e]), xs[a:b].T @ gu[a:b, :F], f"dW1 e{e} (GPU g_bar)", 1e-3, 1e-3)
        assert_wgrad(to_f64(g["dW3"][e]), xs[a:b].T @ gu[a:b, F:], f"dW3 e{e} (GPU u_bar)", 1e-3, 1e-3)
        assert_wgrad(to_f64(g["dW2"][e]), to_f64(hbw[a:b]).T @ ybar[a:b], f"dW2 e{e} (GPU h, y_bar)",
                     1e-3, 1e-3)
    # router pieces from the GPU's own values: w_bar = <d_out, y>, the softmax
    # backward, dWg = x^T l_bar and dbias = column sums of l_bar
    x64, d64 = orc.bf16_to_f64(L["x"]), orc.bf16_to_f64(d_out)
    inv = V["inv"].cpu().numpy().astype(np.int64)
    ids = V["ids"].cpu().numpy().astype(np.int64)
    w32 = V["w"].cpu().numpy().astype(np.float64)
    y_tok = to_f64(V["y"][:S])[inv].reshape(T, k, D)
    wbar, lbar = B["wbar"].cpu().numpy().astype(np.float64), B["lbar"].cpu().numpy().astype(np.float64)
    wbar_ref = np.einsum("td,tjd->tj", d64, y_tok)
    assert_close(wbar, wbar_ref, "w_bar", atol=1e-4 * _rms(wbar_ref), rtol=1e-4)
    lbar_ref = bwd.softmax_backward(w32, wbar)
    assert_close(lbar, lbar_ref, "l_bar", atol=1e-5 * _rms(lbar_ref), rtol=1e-4)
    Ldense = np.zeros((T, E))
    np.put_along_axis(Ldense, ids, lbar, axis=1)
    assert_wgrad(to_f64(g["dWg"]), x64.T @ Ldense, "dWg (GPU l_bar)", 1e-3, 1e-3)
    assert_wgrad(to_f64(g["dbias"]), Ldense.sum(axis=0), "dbias (GPU l_bar)", 1e-3, 1e-3)
    # dx: the gather of the GPU's x_bar rows (+ shared row) + the router term
    xbar_tok = xbar[inv].reshape(T, k, D).sum(axis=1)
    if shared:
        xbar_tok = xbar_tok + to_f64(B["xbar"][Sp:Sp + T])
    dx_ref = xbar_tok + Ldense @ orc.bf16_to_f64(L["Wg"]).T
    assert_close(to_f64(g["dx"]), dx_ref, "dx (GPU x_bar, l_bar)", atol=1e-3 * _rms(dx_ref), rtol=4e-3)
    if shared:
        Ws1, Ws3, Ws2 = (orc.bf16_to_f64(L[n]) for n in ("Ws1", "Ws3", "Ws2"))
        hb_s, gu_s = to_f64(B["hbar"][Sp:Sp + T]), to_f64(B["gu"][Sp:Sp + T])
        assert_close(hb_s, d64 @ Ws2.T, "h_bar shared", atol=H_ATOL, rtol=H_RTOL)
        assert_wgrad(to_f64(g["dWs1"]), x64.T @ gu_s[:, :F], "dWs1 (GPU g_bar)", 1e-3, 1e-3)
        assert_wgrad(to_f64(g["dWs3"]), x64.T @ gu_s[:, F:], "dWs3 (GPU u_bar)", 1e-3, 1e-3)
        assert_wgrad(to_f64(g["dWs2"]), to_f64(V["h"][S:S + T]).T @ d64, "dWs2 (GPU h)", 1e-3, 1e-3)


CASES = [
    # T, D, F, E, k, shared, seed, bias
    (256, 128, 256, 4, 2, False, 40, None),
    (300, 128, 192, 5, 2, True, 41, None),
    (200, 192, 320, 6, 3, True, 42,                    # D, F not multiples of 256; an empty expert
     np.array([0, 0, -1e4, 0, 0, 0], np.float32)),
    (700, 256, 256, 8, 2, False, 43, np.array([3, 2, 0, 0, 0, 0, 0, 0], np.float32)),  # two hot experts
    (64, 64, 64, 16, 4, True, 44, None),               # tiny groups
    (1, 64, 128, 2, 2, True, 45, None),                # one token
    (1100, 384, 512, 4, 1, True, 46, None),            # top-1, several tiles per group
    (12000, 128, 192, 1, 1, True, 49, None),           # routed and shared groups split along their rows
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"T{c[0]}_D{c[1]}_F{c[2]}_E{c[3]}_k{c[4]}_sh{int(c[5])}")
def test_backward_matches_oracle(moe, case):
    T, D, F, E, k, shared, seed, bias = case
    _, L = inputs.make_custom(T, D, F, E, k, shared, seed, bias=bias)
    x64, Wg64 = orc.bf16_to_f64(L["x"]), orc.bf16_to_f64(L["Wg"])
    gap = orc.topk_gap(orc.router_logits(x64, Wg64, L["bias"]), k)
    assert gap.min() > 1e-3, "pick another seed: a token sits near a routing tie"
    d_out = _d_out(T, D, seed)
    _, g, wss = _run(moe, L, k, d_out, shared)
    _stage_checks(moe, L, k, d_out, g, wss, shared)
    ref = bwd.moe_ffn_backward(L["x"], L["Wg"], L["W1"], L["W3"], L["W2"], k, d_out, bias=L["bias"],
                               Ws1=L["Ws1"], Ws3=L["Ws3"], Ws2=L["Ws2"])
    assert_dx(to_f64(g["dx"]), ref["dx"])
    for n in ("dW1", "dW3", "dW2") + (("dWs1", "dWs3", "dWs2") if shared else ()):
        assert_wgrad(to_f64(g[n]), ref[n], n)
    assert_wgrad(to_f64(g["dWg"]), ref["dWg"], "dWg")
    assert_wgrad(to_f64(g["dbias"]), ref["dbias"], "dbias")
    if bias is not None and (bias < -100).any():
        for e in np.nonzero(bias < -100)[0]:      # an expert with no tokens: exactly zero
            assert not g["dW1"][e].any() and not g["dW2"][e].any()


def test_backward_after_chained_forward_and_deterministic(moe):
    T, D, F, E, k = 512, 128, 256, 4, 2
    _, L = inputs.make_custom(T, D, F, E, k, True, 47)
    d_out = _d_out(T, D, 47)
    _, g1, (ws1, _) = _run(moe, L, k, d_out, True)
    _, g2, (_, bws2) = _run(moe, L, k, d_out, True, chained=True)
    for n in g1:
        assert torch.equal(g1[n], g2[n]), n
    # after the chained forward the backward recomputed h itself: the forward's bits
    V, B = ws1.views(), bws2.views()
    prow = torch.tensor(moe.padded_rows(V["counts"].cpu().numpy()), dtype=torch.long, device="cuda")
    assert torch.equal(B["h"][prow], V["h"][:T * k]), "recomputed h differs from the forward's h"
    assert torch.equal(B["h"][B["S_pad"]:B["S_pad"] + T], V["h"][T * k:T * k + T])


def test_backward_fixed_routing_skips_router(moe):
    T, D, F, E, k = 333, 128, 192, 6, 2
    _, L = inputs.make_custom(T, D, F, E, k, False, 48)
    ids, w = orc.topk_softmax(orc.router_logits(orc.bf16_to_f64(L["x"]), orc.bf16_to_f64(L["Wg"])), k)
    d_out = _d_out(T, D, 48)
    _, g, _ = _run(moe, L, k, d_out, False, ids_in=to_dev(ids.astype(np.int32)),
                   weights_in=to_dev(w.astype(np.float32)), router=False)
    ref = bwd.moe_ffn_backward(L["x"], L["Wg"], L["W1"], L["W3"], L["W2"], k, d_out, ids=ids, weights=w)
    assert "dWg" not in g
    assert_dx(to_f64(g["dx"]), ref["dx"], "dx (fixed routing: no router term)")
    for n in ("dW1", "dW3", "dW2"):
        assert_wgrad(to_f64(g[n]), ref[n], n)


@pytest.mark.parametrize("name", ["gptoss_lite", "skewed", "small_chunk", "wide"])
def test_backward_full_size_sampled(moe, name):
    """Full-size workloads with routing fixed from outside: dx on sampled
    tokens and sampled columns of every weight gradient, each computed by the
    oracle from the rows it needs.  skewed adds Zipf load, an empty expert
    (whose gradients must be exactly zero) and groups split along their rows;
    small_chunk adds 64 experts of ~128 rows, top-4 and the shared expert."""
    w_ = inputs.WORKLOADS[name]
    L = inputs.make_layer(w_)
    T, D, F, E, k = w_.T, w_.D, w_.F, w_.E, w_.k
    x64 = orc.bf16_to_f64(L["x"])
    ids, w = orc.topk_softmax(orc.router_logits(x64, orc.bf16_to_f64(L["Wg"]), L["bias"]), k)
    d_out = _d_out(T, D, 5)
    _, g, _ = _run(moe, L, k, d_out, w_.shared, ids_in=to_dev(ids.astype(np.int32)),
                   weights_in=to_dev(w.astype(np.float32)), router=False)
    pm = orc.permutation(ids, E)
    perm, inv, off = pm["perm"].astype(np.int64), pm["inv"].astype(np.int64), pm["offsets"]
    dout64 = orc.bf16_to_f64(d_out)
    rng = np.random.default_rng(3)
    W1, W3, W2 = (orc.bf16_to_f64(L[n]) for n in ("W1", "W3", "W2"))
    # dx on sampled tokens: every slot of the token plus the shared expert
    tokens = np.unique(np.concatenate([rng.choice(T, 48, replace=False), [0, T - 1]]))
    dx_ref = np.zeros((tokens.size, D))
    for i, t in enumerate(tokens):
        for j in range(k):
            e = int(ids[t, j])
            r = bwd.expert_backward(x64[t:t + 1], W1[e], W3[e], W2[e], w[t, j] * dout64[t:t + 1])
            dx_ref[i] += r["xs_bar"][0]
    if w_.shared:
        Ws1, Ws3, Ws2 = (orc.bf16_to_f64(L[n]) for n in ("Ws1", "Ws3", "Ws2"))
        dx_ref += bwd.expert_backward(x64[tokens], Ws1, Ws3, Ws2, dout64[tokens])["xs_bar"]
    assert_dx(to_f64(g["dx"])[tokens], dx_ref, "dx sampled tokens")
    # sampled columns f of dW1[e], dW3[e] and rows f of dW2[e], from the expert's rows
    experts = rng.choice(E, 3, replace=False)
    if w_.empty_expert is not None:
        experts = np.unique(np.append(experts, w_.empty_expert))
    for e in experts:
        a, b = int(off[e]), int(off[e + 1])
        xs = x64[perm[a:b] // k]
        ybar = w[perm[a:b] // k, perm[a:b] % k][:, None] * dout64[perm[a:b] // k]
        for f in rng.choice(F, 2, replace=False):
            gcol, ucol = xs @ W1[e][:, f], xs @ W3[e][:, f]
            hbar = ybar @ W2[e][f, :]
            gb, ub = bwd.swiglu_backward(gcol, ucol, hbar)
            assert_wgrad(to_f64(g["dW1"][e][:, f]), xs.T @ gb, f"dW1[{e}][:, {f}]")
            assert_wgrad(to_f64(g["dW3"][e][:, f]), xs.T @ ub, f"dW3[{e}][:, {f}]")
            hcol = orc.silu(gcol) * ucol
            assert_wgrad(to_f64(g["dW2"][e][f, :]), hcol @ ybar, f"dW2[{e}][{f}, :]")


def test_backward_widest_router_fixed_routing(moe):
    """E = 128 experts (most of them with a handful of rows, some empty) and
    the largest top-k, with the routing fixed from outside."""
    T, D, F, E, k = 300, 128, 128, 128, 16
    _, L = inputs.make_custom(T, D, F, E, k, True, 50)
    ids, w = orc.topk_softmax(orc.router_logits(orc.bf16_to_f64(L["x"]), orc.bf16_to_f64(L["Wg"])), k)
    d_out = _d_out(T, D, 50)
    _, g, _ = _run(moe, L, k, d_out, True, ids_in=to_dev(ids.astype(np.int32)),
                   weights_in=to_dev(w.astype(np.float32)), router=False)
    ref = bwd.moe_ffn_backward(L["x"], L["Wg"], L["W1"], L["W3"], L["W2"], k, d_out, Ws1=L["Ws1"],
                               Ws3=L["Ws3"], Ws2=L["Ws2"], ids=ids, weights=w)
    assert_dx(to_f64(g["dx"]), ref["dx"])
    for n in ("dW1", "dW3", "dW2", "dWs1", "dWs3", "dWs2"):
        assert_wgrad(to_f64(g[n]), ref[n], n)


def test_backward_zero_tokens_is_a_no_op(moe):
    _, L = inputs.make_custom(4, 64, 64, 2, 1, False, 51)
    G = {key: (to_dev(v) if v is not None else None) for key, v in L.items()}
    ws = moe.Workspace(0, 64, 64, 2, 1, False)
    x0 = G["x"][:0]
    g = moe.moe_ffn_backward(x0, G["Wg"], G["W1"], G["W3"], G["W2"], 1, x0, ws)
    assert g["dx"].shape == (0, 64)
