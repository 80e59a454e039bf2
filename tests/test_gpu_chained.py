"""Parity of the chained expert FFN (W1||W3 + SiLU*mul and W2 in one kernel,
h kept on chip) through the C ABI.

* Against the fp64 oracle end to end: y = grouped_down(grouped_swiglu(x_sorted))
  with the layer tolerance |gpu - oracle| <= 1e-2 + 1e-2 |oracle| (the kernel
  rounds h to bf16 between the two products, as the unchained path does).
* Against the oracle's down projection of the separate W1||W3 kernel's bf16 h,
  with the intermediate tolerance: the chained kernel computes h with the same
  fp32 accumulation order and the same SiLU, so only y's rounding remains.
* Bit for bit against the two separate grouped GEMMs (same accumulation
  order, same roundings).
* The whole layer with chained=True against the oracle, and the layer's
  result equal to the unchained layer's.
Shapes: D in {64, 128, 192, 256} (the chained kernel needs D <= 256), ragged
and empty groups, tiny groups, one F chunk, many F chunks, the shared expert.
"""
import numpy as np
import pytest
import torch

from grouped_gemm_router_gb300 import inputs
from oracle import moe_oracle as orc

from _util import assert_close, bf16_bits, to_dev, to_f64

pytestmark = pytest.mark.gpu

H_RTOL, H_ATOL = 4e-3, 1e-4


@pytest.fixture(scope="module")
def moe():
    from grouped_gemm_router_gb300 import build
    build.build()
    from grouped_gemm_router_gb300 import moe as m
    return m


def _routing(L, k, E):
    x, Wg = orc.bf16_to_f64(L["x"]), orc.bf16_to_f64(L["Wg"])
    ids, w = orc.topk_softmax(orc.router_logits(x, Wg, L["bias"]), k)
    pm = orc.permutation(ids, E)
    return ids, w, pm, L["x"][pm["perm"].astype(np.int64) // k]


CASES = [
    # T, D, F, E, k, shared, seed, bias
    (256, 128, 256, 4, 2, False, 20, None),
    (256, 128, 256, 4, 2, True, 21, None),
    (300, 64, 64, 3, 2, True, 22, None),                # D = 64, a single F chunk
    (333, 192, 320, 5, 2, True, 23, None),              # D = 192: W2 halves of 96 columns
    (1000, 256, 1024, 16, 3, False, 24,                  # D = 256, empty experts
     np.array([0, -1e4, 0, 0, 0, -1e4, 0, 0, 0, 0, 0, 0, 0, 0, 0, -1e4], np.float32)),
    (512, 128, 192, 128, 4, True, 25, None),            # 128 tiny groups
    (1, 64, 128, 2, 2, True, 26, None),                 # S = 2 rows
    (700, 256, 512, 8, 2, False, 27, np.array([60, 50, 0, 0, 0, 0, 0, 0], np.float32)),  # hot experts
    (3000, 256, 2048, 8, 2, True, 28, None),            # 32 F chunks, several tiles per group
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"T{c[0]}_D{c[1]}_F{c[2]}_E{c[3]}_k{c[4]}_sh{int(c[5])}")
def test_chained_ffn(moe, case):
    T, D, F, E, k, shared, seed, bias = case
    _, L = inputs.make_custom(T, D, F, E, k, shared, seed, bias=bias)
    _, _, pm, xs_bits = _routing(L, k, E)
    S = T * k
    G = {key: (to_dev(v) if v is not None else None) for key, v in L.items()}
    xs, offs = to_dev(xs_bits), to_dev(pm["offsets"])
    y, ys = moe.moe_grouped_ffn_chained(xs, offs, G["W1"], G["W3"], G["W2"], T, k,
                                        x=G["x"] if shared else None, Ws1=G["Ws1"], Ws3=G["Ws3"], Ws2=G["Ws2"])
    h2 = moe.moe_grouped_swiglu(xs, offs, G["W1"], G["W3"], T, k, x=G["x"] if shared else None,
                                Ws1=G["Ws1"], Ws3=G["Ws3"])
    y2, ys2 = moe.moe_grouped_down(h2, offs, G["W2"], T, k, Ws2=G["Ws2"])
    torch.cuda.synchronize()
    assert moe.device_error() == 0
    y_got = to_f64(y)

    # end to end against the fp64 oracle
    x64 = orc.bf16_to_f64(xs_bits)
    W1, W3, W2 = (orc.bf16_to_f64(L[n]) for n in ("W1", "W3", "W2"))
    y_ref = orc.grouped_down(orc.grouped_swiglu(x64, W1, W3, pm["offsets"]), W2, pm["offsets"])
    assert_close(y_got[:S], y_ref, "y routed vs oracle", atol=1e-2, rtol=1e-2)
    if shared:
        ys_ref = orc.shared_expert(orc.bf16_to_f64(L["x"]), orc.bf16_to_f64(L["Ws1"]),
                                   orc.bf16_to_f64(L["Ws3"]), orc.bf16_to_f64(L["Ws2"]))
        assert_close(to_f64(ys), ys_ref, "ys (shared, fp32) vs oracle", atol=1e-2, rtol=1e-2)

    # the oracle's down projection of the separate kernel's bf16 h
    h_got = to_f64(h2)
    assert_close(y_got[:S], orc.grouped_down(h_got[:S], W2, pm["offsets"]), "y routed", atol=H_ATOL,
                 rtol=H_RTOL)
    if shared:   # fp32 accumulation of the bf16 h and Ws2 products, not rounded to bf16
        assert_close(to_f64(ys), h_got[S:] @ orc.bf16_to_f64(L["Ws2"]), "ys", atol=1e-4, rtol=1e-4)

    # the unchained pair of kernels gives the same bits
    assert torch.equal(y, y2)
    if shared:
        assert torch.equal(ys, ys2)


def test_chained_layer_matches_oracle_and_unchained(moe):
    T, D, F, E, k = 4096, 256, 1024, 8, 2
    _, L = inputs.make_custom(T, D, F, E, k, True, 29)
    G = {key: (to_dev(v) if v is not None else None) for key, v in L.items()}
    args = (G["x"], G["Wg"], G["W1"], G["W3"], G["W2"], k)
    kw = dict(Ws1=G["Ws1"], Ws3=G["Ws3"], Ws2=G["Ws2"])
    n0 = moe.launch_count()
    out_c = moe.moe_ffn_forward(*args, chained=True, **kw)
    n_chained = moe.launch_count() - n0
    out_u = moe.moe_ffn_forward(*args, **kw)
    torch.cuda.synchronize()
    assert moe.device_error() == 0
    assert n_chained == 4    # route (packing its own router weights), scatter, chained FFN, combine
    assert torch.equal(out_c, out_u)
    x64 = orc.bf16_to_f64(L["x"])
    logits = orc.router_logits(x64, orc.bf16_to_f64(L["Wg"]))
    near = orc.topk_gap(logits, k) < 1e-3
    rng = np.random.default_rng(1)
    tokens = np.unique(np.concatenate([rng.choice(T, 512, replace=False), [0, T - 1]]))
    tokens = tokens[~near[tokens]]
    ref = orc.moe_ffn_forward(x64[tokens], L["Wg"], L["W1"], L["W3"], L["W2"], k, Ws1=L["Ws1"],
                              Ws3=L["Ws3"], Ws2=L["Ws2"])
    assert_close(to_f64(out_c)[tokens], ref, "chained layer", atol=1e-2, rtol=1e-2)


def test_chained_full_size_sampled(moe):
    """The largest shape of the chained sweep (T = 32768, D = 256, F = 2048,
    E = 8, top-2): sampled rows, one expert at a time in the oracle, and bit
    equality with the unchained kernels on every row."""
    T, D, F, E, k = 32768, 256, 2048, 8, 2
    _, L = inputs.make_custom(T, D, F, E, k, False, 30)
    _, _, pm, xs_bits = _routing(L, k, E)
    G = {key: (to_dev(v) if v is not None else None) for key, v in L.items()}
    xs, offs = to_dev(xs_bits), to_dev(pm["offsets"])
    y, _ = moe.moe_grouped_ffn_chained(xs, offs, G["W1"], G["W3"], G["W2"], T, k)
    y2, _ = moe.moe_grouped_down(moe.moe_grouped_swiglu(xs, offs, G["W1"], G["W3"], T, k), offs, G["W2"], T, k)
    torch.cuda.synchronize()
    assert moe.device_error() == 0
    assert torch.equal(y, y2)
    S = T * k
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([rng.choice(S, 256, replace=False), pm["offsets"][1:-1],
                                     pm["offsets"][1:-1] - 1, [S - 1]]))
    rows = rows[(rows >= 0) & (rows < S)]
    expert = np.searchsorted(pm["offsets"], rows, side="right") - 1
    y_got = to_f64(y[torch.from_numpy(rows).cuda()])
    for e in np.unique(expert):
        sel = expert == e
        one = np.array([0, int(sel.sum())])
        h = orc.grouped_swiglu(orc.bf16_to_f64(xs_bits[rows[sel]]), orc.bf16_to_f64(L["W1"][e:e + 1]),
                               orc.bf16_to_f64(L["W3"][e:e + 1]), one)
        y_ref = orc.grouped_down(h, orc.bf16_to_f64(L["W2"][e:e + 1]), one)
        assert_close(y_got[sel], y_ref, f"y expert {e}", atol=1e-2, rtol=1e-2)


def test_chained_rejects_wide_rows(moe):
    from grouped_gemm_router_gb300 import _native as N
    _, L = inputs.make_custom(64, 320, 64, 2, 1, False, 31)
    G = {key: (to_dev(v) if v is not None else None) for key, v in L.items()}
    with pytest.raises(N.MoeError) as ei:
        moe.moe_ffn_forward(G["x"], G["Wg"], G["W1"], G["W3"], G["W2"], 1, chained=True)
    assert ei.value.status == N.MOE_ERR_UNSUPPORTED_SHAPE
