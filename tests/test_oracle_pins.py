"""Pins for the fp64 oracle, independent of the oracle's own code.

Each test checks the oracle against something the pages or the mathematics
fix: a brute-force dense evaluation written here with plain Python loops, a
printed number from the pages (tests/golden/), closed forms, invariants and
special cases.  None of these re-types the oracle's formulas through the same
library calls.
"""
import json
import math
import os
import random

import numpy as np
import pytest

from oracle import moe_oracle as orc
from grouped_gemm_router_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------
# Independent brute force, plain Python: every token through every expert,
# masked by the routing decision (no permutation, no grouping).
# ----------------------------------------------------------------------------
def _py_bf16(bits):
    """bf16 bits -> float via the IEEE bit layout (struct), independent of numpy views."""
    import struct
    return struct.unpack("<f", struct.pack("<I", int(bits) << 16))[0]


def _to_py(a):
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return np.vectorize(_py_bf16, otypes=[float])(a).tolist()
    return a.astype(float).tolist()


def _py_swiglu(xrow, W1, W3, W2):
    D, F = len(W1), len(W1[0])
    h = []
    for f in range(F):
        g = sum(xrow[d] * W1[d][f] for d in range(D))
        u = sum(xrow[d] * W3[d][f] for d in range(D))
        sig = 1.0 / (1.0 + math.exp(-g)) if g > -700 else 0.0
        h.append(g * sig * u)
    Dout = len(W2[0])
    return [sum(h[f] * W2[f][d] for f in range(F)) for d in range(Dout)]


def brute_force_layer(x, Wg, W1, W3, W2, k, bias=None, Ws1=None, Ws3=None, Ws2=None):
    x, Wg, W1, W3, W2 = map(_to_py, (x, Wg, W1, W3, W2))
    shared = Ws1 is not None
    if shared:
        Ws1, Ws3, Ws2 = map(_to_py, (Ws1, Ws3, Ws2))
    T, D, E = len(x), len(x[0]), len(W1)
    b = [0.0] * E if bias is None else [float(v) for v in bias]
    out, all_ids, all_w = [], [], []
    for t in range(T):
        logits = [sum(x[t][d] * Wg[d][e] for d in range(D)) + b[e] for e in range(E)]
        ranked = sorted(range(E), key=lambda e: (-logits[e], e))
        chosen = ranked[:k]
        m = logits[chosen[0]]
        z = [math.exp(logits[e] - m) for e in chosen]
        gate = {e: z[i] / sum(z) for i, e in enumerate(chosen)}
        acc = [0.0] * D
        for e in range(E):
            weight = gate.get(e, 0.0)          # dense evaluation, masked
            y = _py_swiglu(x[t], W1[e], W3[e], W2[e])
            for d in range(D):
                acc[d] += weight * y[d]
        if shared:
            ys = _py_swiglu(x[t], Ws1, Ws3, Ws2)
            acc = [acc[d] + ys[d] for d in range(D)]
        out.append(acc)
        all_ids.append(chosen)
        all_w.append([gate[e] for e in chosen])
    return np.array(out), np.array(all_ids), np.array(all_w)


def _tiny(T=24, D=8, F=12, E=5, k=2, shared=True, seed=11, bias=None):
    w, layer = inputs.make_custom(T, D, F, E, k, shared, seed, bias=bias)
    return w, layer


def _run_oracle(w, L, **kw):
    return orc.moe_ffn_forward(L["x"], L["Wg"], L["W1"], L["W3"], L["W2"], w.k,
                               bias=L["bias"], Ws1=L["Ws1"], Ws3=L["Ws3"], Ws2=L["Ws2"],
                               return_all=True, **kw)


# ----------------------------------------------------------------------------
# bf16 widening and silu: values fixed by the formats / the definition
# ----------------------------------------------------------------------------
def test_bf16_widening_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x3EAA, 0x7F7F, 0x0001], dtype=np.uint16)
    want = [1.0, -2.0, 0.0, -0.0, 0.33203125, 3.3895313892515355e38, 2.0 ** -133]
    got = orc.bf16_to_f64(bits)
    assert got.dtype == np.float64
    for g, v in zip(got, want):
        assert g == v


def test_silu_closed_forms():
    z = np.array([0.0, 1.0, -1.0, 2.5, -30.0, 40.0, -800.0])
    s = orc.silu(z)
    assert s[0] == 0.0
    assert s[1] == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)
    # silu(z) - silu(-z) = z because sigmoid(z) + sigmoid(-z) = 1
    assert s[1] - s[2] == pytest.approx(1.0, rel=1e-15)
    assert s[5] == pytest.approx(40.0, rel=1e-15)        # sigmoid(40) == 1 in fp64
    assert abs(s[4]) < 1e-11 and s[4] < 0
    assert s[6] == 0.0                                    # no overflow to nan


# ----------------------------------------------------------------------------
# Routing: brute force, special cases, textbook softmax
# ----------------------------------------------------------------------------
def test_topk_softmax_brute_force_with_ties():
    rng = random.Random(5)
    T, E, k = 200, 9, 3
    # coarse values so that exact ties are frequent
    logits = np.array([[rng.choice([-1.0, -0.5, 0.0, 0.25, 0.5, 2.0]) for _ in range(E)]
                       for _ in range(T)])
    ids, w = orc.topk_softmax(logits, k)
    for t in range(T):
        ranked = sorted(range(E), key=lambda e: (-logits[t, e], e))[:k]
        assert ids[t].tolist() == ranked
        z = [math.exp(logits[t, e]) for e in ranked]
        for j in range(k):
            assert w[t, j] == pytest.approx(z[j] / sum(z), rel=1e-14)


def test_zero_router_gives_first_k_experts_and_uniform_weights():
    T, E, k = 7, 6, 4
    ids, w = orc.topk_softmax(np.zeros((T, E)), k)
    assert (ids == np.arange(k)[None, :]).all()
    assert (w == 1.0 / k).all()


def test_k_equals_E_is_full_softmax():
    from scipy.special import softmax
    rng = np.random.default_rng(3)
    logits = rng.normal(size=(10, 6))
    ids, w = orc.topk_softmax(logits, 6)
    full = softmax(logits, axis=1)
    assert np.allclose(np.take_along_axis(full, ids.astype(np.int64), 1), w, rtol=1e-14, atol=0)
    assert (np.diff(np.take_along_axis(logits, ids.astype(np.int64), 1), axis=1) <= 0).all()


def test_one_hot_bias_forces_experts():
    w_, L = _tiny(T=10, E=6, k=2, shared=False)
    bias = np.array([0, 0, 100, 0, 50, 0], dtype=np.float32)
    x, Wg = orc.bf16_to_f64(L["x"]), orc.bf16_to_f64(L["Wg"])
    ids, w = orc.topk_softmax(orc.router_logits(x, Wg, bias), 2)
    assert (ids[:, 0] == 2).all() and (ids[:, 1] == 4).all()
    xs, Wgs = _to_py(L["x"]), _to_py(L["Wg"])
    for t in range(10):
        l2 = sum(xs[t][d] * Wgs[d][2] for d in range(len(Wgs))) + 100.0
        l4 = sum(xs[t][d] * Wgs[d][4] for d in range(len(Wgs))) + 50.0
        assert w[t, 1] == pytest.approx(1.0 / (1.0 + math.exp(l2 - l4)), rel=1e-9)


def test_gate_weights_sum_to_one():
    w_, L = _tiny(T=64, E=8, k=3)
    r = _run_oracle(w_, L)
    assert np.abs(r["w"].sum(axis=1) - 1.0).max() < 1e-15
    assert (r["w"] > 0).all()
    assert (np.diff(r["w"], axis=1) <= 0).all()        # descending logits -> descending weights


def test_topk_gap():
    logits = np.array([[3.0, 1.0, 2.0, 0.5], [1.0, 1.0, 1.0, 1.0]])
    assert orc.topk_gap(logits, 2).tolist() == [1.0, 0.0]
    assert np.isinf(orc.topk_gap(logits, 4)).all()


# ----------------------------------------------------------------------------
# Permutation: invariants and brute force
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("E,k,T", [(4, 2, 50), (8, 2, 333), (64, 4, 90), (3, 3, 17), (1, 1, 5)])
def test_permutation_invariants_and_brute_force(E, k, T):
    rng = random.Random(E * 1000 + T)
    ids = np.array([rng.sample(range(E), k) for _ in range(T)], dtype=np.int32)
    pm = orc.permutation(ids, E)
    S = T * k
    flat = ids.reshape(-1)
    perm, inv, counts, offsets = pm["perm"], pm["inv"], pm["counts"], pm["offsets"]
    assert counts.sum() == S and offsets[0] == 0 and offsets[-1] == S
    assert (np.diff(offsets) == counts).all()
    assert sorted(perm.tolist()) == list(range(S))                 # bijection
    assert (inv[perm] == np.arange(S)).all() and (perm[inv] == np.arange(S)).all()
    brute = sorted(range(S), key=lambda s: (int(flat[s]), s))       # stable by slot
    assert perm.tolist() == brute
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert (flat[seg] == e).all() and (np.diff(seg) > 0).all()
        assert counts[e] == sum(1 for s in range(S) if flat[s] == e)


def test_gather_is_repeat_interleave_then_permute():
    x = np.arange(12.0).reshape(4, 3)
    perm = np.array([3, 0, 7, 5, 1, 2, 4, 6])
    xs = orc.gather_sorted(x, perm, 2)
    rep = np.concatenate([[x[t]] * 2 for t in range(4)])            # repeat_interleave by hand
    assert (xs == rep[perm]).all()


# ----------------------------------------------------------------------------
# Whole layer vs brute-force dense masked evaluation
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("T,D,F,E,k,shared,seed", [
    (24, 8, 12, 5, 2, True, 11),
    (16, 16, 8, 4, 2, False, 12),
    (9, 8, 16, 8, 3, True, 13),
    (12, 8, 8, 3, 3, False, 14),     # k == E: every expert on every token
])
def test_layer_matches_dense_masked_brute_force(T, D, F, E, k, shared, seed):
    w_, L = _tiny(T, D, F, E, k, shared, seed)
    r = _run_oracle(w_, L)
    bf_out, bf_ids, bf_w = brute_force_layer(L["x"], L["Wg"], L["W1"], L["W3"], L["W2"], k,
                                             L["bias"], L["Ws1"], L["Ws3"], L["Ws2"])
    assert (r["ids"] == bf_ids).all()
    assert np.allclose(r["w"], bf_w, rtol=1e-13, atol=0)
    assert np.abs(r["out"] - bf_out).max() <= 1e-12 * max(1.0, np.abs(bf_out).max())


def test_empty_expert_is_skipped_and_layer_still_exact():
    bias = np.array([0, 0, -1e4, 0, 0], dtype=np.float32)
    w_, L = _tiny(T=20, D=8, F=8, E=5, k=2, shared=False, seed=21, bias=bias)
    r = _run_oracle(w_, L)
    assert r["counts"][2] == 0 and r["offsets"][2] == r["offsets"][3]
    bf_out, _, _ = brute_force_layer(L["x"], L["Wg"], L["W1"], L["W3"], L["W2"], 2, bias)
    assert np.abs(r["out"] - bf_out).max() <= 1e-12


def test_single_expert_top1_is_dense_swiglu():
    """E = 1, k = 1: the router always picks expert 0 with weight 1, so the
    layer is the dense SwiGLU FFN W2(silu(x W1) * (x W3))."""
    w_, L = _tiny(T=6, D=8, F=8, E=1, k=1, shared=False, seed=31)
    r = _run_oracle(w_, L)
    x, W1, W3, W2 = map(_to_py, (L["x"], L["W1"][0], L["W3"][0], L["W2"][0]))
    for t in range(6):
        want = _py_swiglu(x[t], W1, W3, W2)
        assert np.allclose(r["out"][t], want, rtol=1e-13, atol=1e-15)
    assert (r["w"] == 1.0).all()


def test_fixed_routing_path_equals_own_routing():
    w_, L = _tiny(T=30, E=6, k=2, shared=True, seed=41)
    r = _run_oracle(w_, L)
    r2 = _run_oracle(w_, L, ids=r["ids"], weights=r["w"])
    assert (r2["out"] == r["out"]).all()


# ----------------------------------------------------------------------------
# Numbers printed on the pages
# ----------------------------------------------------------------------------
def test_w1w3_flop_count_matches_page():
    g = json.load(open(os.path.join(GOLDEN, "p1_w1w3_flops.json")))
    flops = orc.w1w3_flops(g["tokens"], g["d_model"], g["d_ff"], g["top_k"])
    assert flops == 309_237_645_312
    assert round(flops / 1e9) == g["gflop_printed"]


class _MacCounter:
    """Plain-Python evaluation of the layer that counts every multiply-add it
    performs.  Only the experts a token is routed to are evaluated (the
    'active' work), unlike the dense masked brute force above; the output is
    returned so that the counted evaluation can be checked for correctness."""

    def __init__(self):
        self.macs = 0

    def dot(self, a, b):
        self.macs += len(a)
        return sum(p * q for p, q in zip(a, b))

    def vecmat(self, v, M):                # v [n] @ M [n][m]
        return [self.dot(v, [M[i][j] for i in range(len(M))]) for j in range(len(M[0]))]

    def swiglu(self, xrow, W1, W3, W2):
        g, u = self.vecmat(xrow, W1), self.vecmat(xrow, W3)
        h = [gi / (1.0 + math.exp(-gi)) * ui for gi, ui in zip(g, u)]
        return self.vecmat(h, W2)

    def layer(self, x, Wg, W1, W3, W2, k, Ws1=None, Ws3=None, Ws2=None):
        x, Wg, W1, W3, W2 = map(_to_py, (x, Wg, W1, W3, W2))
        out = []
        for t in range(len(x)):
            logits = self.vecmat(x[t], Wg)
            chosen = sorted(range(len(W1)), key=lambda e: (-logits[e], e))[:k]
            z = [math.exp(logits[e] - logits[chosen[0]]) for e in chosen]
            acc = [0.0] * len(x[t])
            for e, ze in zip(chosen, z):
                y = self.swiglu(x[t], W1[e], W3[e], W2[e])
                acc = [a + ze / sum(z) * yi for a, yi in zip(acc, y)]
            if Ws1 is not None:
                ys = self.swiglu(x[t], *map(_to_py, (Ws1, Ws3, Ws2)))
                acc = [a + yi for a, yi in zip(acc, ys)]
            out.append(acc)
        return np.array(out)


@pytest.mark.parametrize("T,D,F,E,k,shared", [(6, 8, 12, 5, 2, True), (5, 16, 8, 7, 3, False),
                                              (4, 8, 8, 3, 3, True)])
def test_active_flops_equals_counted_multiply_adds(T, D, F, E, k, shared):
    """active_flops = 2 x the multiply-adds a sparse evaluation of the layer
    actually performs (router, the k routed experts per token, the shared
    expert).  A wrong router, routed or shared term changes the count."""
    w_, L = _tiny(T, D, F, E, k, shared, seed=71 + T)
    mc = _MacCounter()
    got = mc.layer(L["x"], L["Wg"], L["W1"], L["W3"], L["W2"], k, L["Ws1"], L["Ws3"], L["Ws2"])
    ref = _run_oracle(w_, L)["out"]
    assert np.abs(got - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())   # the counted run is the layer
    assert orc.active_flops(T, D, F, E, k, shared) == 2 * mc.macs
    # the routed W1 and W3 products alone are the page's W1/W3 stage count
    mc13 = _MacCounter()
    xs, W1s, W3s = _to_py(L["x"]), _to_py(L["W1"]), _to_py(L["W3"])
    for t in range(T):
        for e in range(k):                     # any k experts: the count does not depend on which
            mc13.vecmat(xs[t], W1s[e])
            mc13.vecmat(xs[t], W3s[e])
    assert orc.w1w3_flops(T, D, F, k) == 2 * mc13.macs


def test_activation_traffic_saving_matches_page(monkeypatch):
    """Part A section 6.2 of the Triton-MoE page: fusing W1/W3 with silu*mul
    removes four activation streams (write g, write u, read g, read u) of
    bf16 [slots, d_ff] tensors, 96 MiB for 4096 tokens x top-2 at d_ff = 1536.
    The element counts are taken from the oracle's own g and u intermediates
    at that shape (d_model does not enter them, so a small one is used)."""
    g = json.load(open(os.path.join(GOLDEN, "p1_activation_traffic.json")))
    T, k, E, F, D = g["slots"] // 2, 2, 8, g["d_ff"], 8
    assert T * k == g["slots"]
    rng = np.random.default_rng(0)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    pm = orc.permutation(ids, E)
    x = rng.standard_normal((T, D))
    xs = orc.gather_sorted(x, pm["perm"], k)
    W1, W3 = rng.standard_normal((E, D, F)), rng.standard_normal((E, D, F))
    seen = []
    real_silu = orc.silu

    def recording_silu(z):             # silu is applied to g, one expert's [rows, F] block at a time
        seen.append(z.size)
        return real_silu(z)
    monkeypatch.setattr(orc, "silu", recording_silu)
    h = orc.grouped_swiglu(xs, W1, W3, pm["offsets"])
    g_elems = sum(seen)
    u_elems = h.size                   # u has the shape of h (and of g)
    assert g_elems == u_elems == g["slots"] * g["d_ff"]
    streams = 2 * g_elems + 2 * u_elems          # write g, write u, read g, read u
    saved = streams * g["bytes_per_element"]
    assert g["streams_removed"] == 4
    assert saved == g["mib_printed"] * 2 ** 20


# ----------------------------------------------------------------------------
# Planted mistakes: each must be caught by the brute-force pin
# ----------------------------------------------------------------------------
def _swap_w1_w3(mp):
    f = orc.grouped_swiglu
    mp.setattr(orc, "grouped_swiglu", lambda xs, W1, W3, off: f(xs, W3, W1, off))


def _softmax_over_all_experts(mp):
    f = orc.topk_softmax

    def g(lg, k):
        ids, _ = f(lg, k)
        full = np.exp(lg) / np.exp(lg).sum(axis=1, keepdims=True)
        return ids, np.take_along_axis(full, ids.astype(np.int64), axis=1)
    mp.setattr(orc, "topk_softmax", g)


def _ties_to_higher_index(mp):
    f = orc.topk_softmax

    def g(lg, k):
        ids, w = f(lg[:, ::-1], k)
        return (lg.shape[1] - 1 - ids).astype(np.int32), w
    mp.setattr(orc, "topk_softmax", g)


def _inverse_swapped_for_forward(mp):
    f = orc.combine
    mp.setattr(orc, "combine", lambda y, inv, w, ys=None: f(y, np.argsort(inv), w, ys))


MUTATIONS = {
    "swap_w1_w3": _swap_w1_w3,
    "softmax_over_all_experts": _softmax_over_all_experts,
    "plain_silu_no_gate": lambda mp: mp.setattr(orc, "silu", lambda z: z),
    "drop_shared": lambda mp: mp.setattr(orc, "shared_expert",
                                         lambda x, a, b, c: np.zeros((x.shape[0], c.shape[1]))),
    "forward_perm_instead_of_inverse": _inverse_swapped_for_forward,
    "ties_to_higher_index": _ties_to_higher_index,
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistakes_are_caught(name, monkeypatch):
    w_, L = _tiny(T=16, D=8, F=8, E=4, k=2, shared=True, seed=51)
    L = dict(L)
    L["Wg"] = L["Wg"].copy()
    L["Wg"][:, 2] = L["Wg"][:, 1]                    # experts 1 and 2 always tie
    bf_out, bf_ids, _ = brute_force_layer(L["x"], L["Wg"], L["W1"], L["W3"], L["W2"], 2,
                                          None, L["Ws1"], L["Ws3"], L["Ws2"])
    clean = _run_oracle(w_, L)
    assert np.abs(clean["out"] - bf_out).max() <= 1e-12 and (clean["ids"] == bf_ids).all()
    MUTATIONS[name](monkeypatch)
    bad = _run_oracle(w_, L)
    assert np.abs(bad["out"] - bf_out).max() > 1e-6 or (bad["ids"] != bf_ids).any()


# ----------------------------------------------------------------------------
# Input generator (no arithmetic of the layer): determinism and rounding
# ----------------------------------------------------------------------------
def test_inputs_deterministic_and_rne():
    w = inputs.WORKLOADS["tiny"]
    a, b = inputs.make_layer(w), inputs.make_layer(w)
    for key in ("x", "Wg", "W1", "W3", "W2"):
        assert (a[key] == b[key]).all()
    assert a["x"].shape == (256, 128) and a["W1"].shape == (4, 128, 256) and a["W2"].shape == (4, 256, 128)
    # round-to-nearest-even on hand-picked float32 values
    f = np.array([1.0, 1.00390625, 1.01171875, 1.0000001, -3.0], dtype=np.float32)
    assert inputs.f32_to_bf16_bits(f).tolist() == [0x3F80, 0x3F80, 0x3F82, 0x3F80, 0xC040]


def test_skewed_bias():
    b = inputs.zipf_router_bias(8, 1.2, 7)
    assert b[7] == np.float32(-1e4)
    p = np.exp(b[:7].astype(np.float64))
    assert abs(p.sum() - 1) < 1e-6 and (np.diff(p) < 0).all()
    assert p[0] / p[1] == pytest.approx(2 ** 1.2, rel=1e-5)
