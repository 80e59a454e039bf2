"""Stage-by-stage parity of the CUDA path (through the C ABI) with the fp64
oracle: routing, permutation (bit-exact), the two grouped GEMMs and the
combine, on small multi-tile shapes with ragged groups, empty experts and the
degenerate cases, and on the full-size workloads."""
import numpy as np
import pytest
import torch

from grouped_gemm_router_gb300 import inputs
from oracle import moe_oracle as orc

from _util import assert_close, bf16_bits, to_dev, to_f64

pytestmark = pytest.mark.gpu

# Intermediates h and y are rounded once to bf16 after fp32 accumulation of
# exact bf16 products: |err| <= 2^-9 |ref| plus fp32 summation noise.
H_RTOL, H_ATOL = 4e-3, 1e-4


@pytest.fixture(scope="module")
def moe():
    from grouped_gemm_router_gb300 import build
    build.build()
    from grouped_gemm_router_gb300 import moe as m
    return m


def _layer(T, D, F, E, k, shared, seed, bias=None):
    return inputs.make_custom(T, D, F, E, k, shared, seed, bias=bias)


def _oracle_routing(L, k):
    x, Wg = orc.bf16_to_f64(L["x"]), orc.bf16_to_f64(L["Wg"])
    logits = orc.router_logits(x, Wg, L["bias"])
    ids, w = orc.topk_softmax(logits, k)
    return logits, ids, w, orc.topk_gap(logits, k)


ROUTE_CASES = [
    # T, D, F, E, k, shared, seed, bias
    (256, 128, 256, 4, 2, False, 0, None),
    (1000, 256, 64, 8, 2, False, 1, None),
    (1, 64, 64, 3, 1, False, 2, None),
    (333, 192, 64, 20, 5, False, 3, None),          # E padded to 24
    (300, 512, 64, 64, 4, False, 4, None),
    (200, 384, 64, 128, 16, False, 5, None),        # widest router, largest k
    (257, 4608, 64, 8, 2, False, 6, None),          # long D: 6 stages per 16-token tile
    (500, 768, 64, 8, 2, False, 7, inputs.zipf_router_bias(8, 1.2, 7)),
    (12000, 768, 64, 8, 2, False, 8, None),         # 32-token blocks
    (20000, 256, 64, 16, 2, False, 9, None),        # 64-token blocks
    (40000, 2048, 64, 16, 2, False, 10, None),      # 4 stages per tile, ~16 tiles per CTA
    (3000, 2048, 64, 128, 8, False, 11, None),      # router weights too large to stage in smem
]


@pytest.mark.parametrize("case", ROUTE_CASES, ids=lambda c: f"T{c[0]}_D{c[1]}_E{c[3]}_k{c[4]}")
def test_route(moe, case):
    T, D, F, E, k, shared, seed, bias = case
    w_, L = _layer(T, D, F, E, k, shared, seed, bias)
    logits, ids_ref, w_ref, gap = _oracle_routing(L, k)
    ids, w, hist = moe.moe_route(to_dev(L["x"]), to_dev(L["Wg"]), k,
                                 bias=to_dev(L["bias"]) if L["bias"] is not None else None)
    torch.cuda.synchronize()
    ids, w, hist = ids.cpu().numpy(), w.cpu().numpy(), hist.cpu().numpy()
    near = gap < 1e-3
    mism = (ids != ids_ref).any(axis=1)
    assert not (mism & ~near).any(), f"{int((mism & ~near).sum())} tokens differ outside the near-tie window"
    ok = ~mism
    assert np.abs(w[ok] - w_ref[ok]).max() < 1e-4
    assert np.abs(w.sum(axis=1) - 1).max() < 1e-5
    from grouped_gemm_router_gb300 import _native
    tb = int(_native.lib.moe_route_block_tokens(T))
    assert hist.shape[0] == (T + tb - 1) // tb
    for b in range(hist.shape[0]):  # per-block histogram of the GPU's own ids
        blk = ids[b * tb:(b + 1) * tb].reshape(-1)
        assert (hist[b] == np.bincount(blk, minlength=E)).all()


def test_route_block_tokens_follow_the_sm_count(moe):
    """64-token blocks when that still gives every SM two of them, else 32 or 16."""
    from grouped_gemm_router_gb300 import _native
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for T in (1, 2048, 32 * 2 * sms - 1, 32 * 2 * sms, 64 * 2 * sms - 1, 64 * 2 * sms, 32768, 1 << 20):
        want = 64 if T >= 64 * 2 * sms else 32 if T >= 32 * 2 * sms else 16
        assert int(_native.lib.moe_route_block_tokens(T)) == want, T


def test_route_all_ties_pick_lowest_experts(moe):
    T, D, E, k = 130, 128, 8, 3
    x = to_dev(inputs.f32_to_bf16_bits(np.random.default_rng(0).normal(size=(T, D)).astype(np.float32)))
    Wg = torch.zeros(D, E, dtype=torch.bfloat16, device="cuda")
    ids, w, _ = moe.moe_route(x, Wg, k)
    assert (ids.cpu().numpy() == np.arange(k)).all()
    assert (w.cpu().numpy() == np.float32(1.0 / 3.0)).all()


PERM_CASES = [
    # T, E, k, distribution
    (1, 1, 1, "uniform"), (63, 8, 2, "uniform"), (64, 8, 2, "uniform"), (65, 8, 2, "uniform"),
    (1000, 8, 2, "uniform"), (300, 128, 16, "uniform"), (777, 5, 3, "one_expert_heavy"),
    (4096, 16, 2, "zipf_with_empty"), (32768, 8, 2, "uniform"), (2048, 64, 4, "uniform"),
]


def _ids(T, E, k, dist, seed):
    rng = np.random.default_rng(seed)
    if dist == "uniform":
        return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    if dist == "one_expert_heavy":
        out = np.stack([rng.permutation(E)[:k] for _ in range(T)])
        out[:, 0] = 2
        out[:, 1:] = np.where(out[:, 1:] == 2, 4, out[:, 1:])
        return out.astype(np.int32)
    p = np.array([(e + 1) ** -1.2 for e in range(E)])
    p[E - 1] = 0
    p /= p.sum()
    return np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("case", PERM_CASES, ids=lambda c: f"T{c[0]}_E{c[1]}_k{c[2]}_{c[3]}")
def test_permute_bit_exact(moe, case):
    T, E, k, dist = case
    ids = _ids(T, E, k, dist, T + E)
    D = 128
    x = inputs.f32_to_bf16_bits(np.random.default_rng(T).normal(size=(T, D)).astype(np.float32))
    r = moe.moe_permute(to_dev(ids), E, x=to_dev(x))
    torch.cuda.synchronize()
    ref = orc.permutation(ids, E)
    for key in ("counts", "offsets", "perm", "inv"):
        got = r[key].cpu().numpy()
        assert (got == ref[key]).all(), f"{key} differs"
    xs = bf16_bits(r["x_sorted"])
    assert (xs == x[ref["perm"] // k]).all()


def _grouped_inputs(L, k, E):
    _, ids, w, _ = _oracle_routing(L, k)
    pm = orc.permutation(ids, E)
    xs_bits = L["x"][pm["perm"].astype(np.int64) // k]
    return ids, w, pm, xs_bits


GEMM_CASES = [
    # T, D, F, E, k, shared, seed, bias
    (256, 128, 256, 4, 2, False, 10, None),
    (256, 128, 256, 4, 2, True, 11, None),
    (300, 192, 192, 5, 2, True, 12, None),            # 64-wide tiles on both GEMMs
    (1000, 384, 640, 16, 3, False, 13, np.array([0, -1e4, 0, 0, 0, -1e4, 0, 0, 0, 0, 0, 0, 0, 0, 0, -1e4], np.float32)),
    (512, 256, 256, 128, 4, True, 14, None),           # 128 tiny groups
    (1, 64, 64, 2, 2, True, 15, None),                # S = 2 rows, smaller than one tile
    (700, 128, 128, 8, 2, False, 16, np.array([60, 50, 0, 0, 0, 0, 0, 0], np.float32)),  # two hot experts
    (2048, 768, 1536, 64, 4, True, 3, None),          # small-chunk shape
    (640, 2048, 1024, 4, 1, False, 17, None),         # long K (32 k-blocks)
]


@pytest.mark.parametrize("case", GEMM_CASES, ids=lambda c: f"T{c[0]}_D{c[1]}_F{c[2]}_E{c[3]}_k{c[4]}_sh{int(c[5])}")
def test_grouped_gemms(moe, case):
    T, D, F, E, k, shared, seed, bias = case
    w_, L = _layer(T, D, F, E, k, shared, seed, bias)
    ids, w, pm, xs_bits = _grouped_inputs(L, k, E)
    offs = to_dev(pm["offsets"])
    h = moe.moe_grouped_swiglu(to_dev(xs_bits), offs, to_dev(L["W1"]), to_dev(L["W3"]), T, k,
                               x=to_dev(L["x"]) if shared else None,
                               Ws1=to_dev(L["Ws1"]), Ws3=to_dev(L["Ws3"]))
    torch.cuda.synchronize()
    S = T * k
    h_ref = orc.grouped_swiglu(orc.bf16_to_f64(xs_bits), orc.bf16_to_f64(L["W1"]),
                               orc.bf16_to_f64(L["W3"]), pm["offsets"])
    h_got = to_f64(h)
    assert_close(h_got[:S], h_ref, "h (routed)", atol=H_ATOL, rtol=H_RTOL)
    if shared:
        x64 = orc.bf16_to_f64(L["x"])
        hs_ref = orc.silu(x64 @ orc.bf16_to_f64(L["Ws1"])) * (x64 @ orc.bf16_to_f64(L["Ws3"]))
        assert_close(h_got[S:], hs_ref, "h (shared)", atol=H_ATOL, rtol=H_RTOL)
    # down projection on the GPU's own (bf16) h
    y, ys = moe.moe_grouped_down(h, offs, to_dev(L["W2"]), T, k, Ws2=to_dev(L["Ws2"]))
    torch.cuda.synchronize()
    y_ref = orc.grouped_down(h_got[:S], orc.bf16_to_f64(L["W2"]), pm["offsets"])
    y_got = to_f64(y)
    assert_close(y_got, y_ref, "y (routed)", atol=H_ATOL, rtol=H_RTOL)
    ys_got = to_f64(ys) if shared else None
    if shared:   # fp32 accumulation of the bf16 h and Ws2 products, not rounded to bf16
        assert_close(ys_got, h_got[S:] @ orc.bf16_to_f64(L["Ws2"]), "ys (shared)", atol=1e-4, rtol=1e-4)
    # combine on the GPU's own y and ys
    out = moe.moe_combine(y, to_dev(w.astype(np.float32)), to_dev(pm["inv"]), ys=ys)
    torch.cuda.synchronize()
    out_ref = orc.combine(y_got, pm["inv"], w.astype(np.float32).astype(np.float64), ys_got)
    assert_close(to_f64(out), out_ref, "combine", atol=1e-3, rtol=4e-3)
    assert moe.device_error() == 0


@pytest.mark.parametrize("D", [192, 256])
def test_expert_weights_do_not_reach_other_experts(moe, D):
    """Each expert's h depends on its own W1 / W3 rows only: with an inf in
    every row of the next expert's W1 and W3, the rows of expert 0 still match
    the oracle (D = 192 is not a multiple of the 128-deep W1||W3 stage, so it
    stages 64 k; D = 256 stages 128 k)."""
    T, F, E, k = 300, 256, 4, 2
    w_, L = _layer(T, D, F, E, k, False, 18)
    ids, w, pm, xs_bits = _grouped_inputs(L, k, E)
    W1, W3 = L["W1"].copy(), L["W3"].copy()
    inf_bits = np.uint16(0x7F80)  # bf16 +inf
    W1[1, :, 0] = inf_bits
    W3[1, :, 0] = inf_bits
    h = moe.moe_grouped_swiglu(to_dev(xs_bits), to_dev(pm["offsets"]), to_dev(W1), to_dev(W3), T, k)
    torch.cuda.synchronize()
    o0, o1 = int(pm["offsets"][0]), int(pm["offsets"][1])
    assert o1 > o0
    h_ref = orc.grouped_swiglu(orc.bf16_to_f64(xs_bits[o0:o1]), orc.bf16_to_f64(L["W1"][:1]),
                               orc.bf16_to_f64(L["W3"][:1]), np.array([0, o1 - o0], dtype=np.int64))
    h0 = to_f64(h)[o0:o1]
    assert np.isfinite(h0).all()
    assert_close(h0, h_ref, "h of expert 0", atol=H_ATOL, rtol=H_RTOL)


def test_combine_exact_small(moe):
    """Combine with y values and weights that are exact in bf16/fp32: the
    fp32 sum is exact, so the bf16 output equals the rounded fp64 sum."""
    T, D, k = 70, 64, 3
    rng = np.random.default_rng(1)
    S = T * k
    y = (rng.integers(-64, 64, size=(S, D)) / 16.0).astype(np.float32)
    ys = (rng.integers(-4096, 4096, size=(T, D)) / 1024.0).astype(np.float32)   # exact in fp32, not in bf16
    perm = rng.permutation(S).astype(np.int32)
    inv = np.empty(S, np.int32)
    inv[perm] = np.arange(S, dtype=np.int32)
    w = (rng.integers(1, 8, size=(T, k)) / 8.0).astype(np.float32)
    out = moe.moe_combine(to_dev(inputs.f32_to_bf16_bits(y)), to_dev(w), to_dev(inv), ys=to_dev(ys))
    ref = orc.combine(y.astype(np.float64), inv, w.astype(np.float64), ys.astype(np.float64))
    assert (bf16_bits(out) == inputs.f32_to_bf16_bits(ref.astype(np.float32))).all()


@pytest.mark.parametrize("name", ["gptoss_lite", "wide"])
def test_grouped_gemms_full_size_sampled(moe, name):
    """Full-size grouped GEMMs (the launch configuration of the benchmark),
    checked on sampled rows that the oracle computes one expert at a time."""
    w_ = inputs.WORKLOADS[name]
    L = inputs.make_layer(w_)
    T, D, F, E, k = w_.T, w_.D, w_.F, w_.E, w_.k
    ids, w, pm, xs_bits = _grouped_inputs(L, k, E)
    offs = to_dev(pm["offsets"])
    h = moe.moe_grouped_swiglu(to_dev(xs_bits), offs, to_dev(L["W1"]), to_dev(L["W3"]), T, k,
                               x=to_dev(L["x"]) if w_.shared else None,
                               Ws1=to_dev(L["Ws1"]), Ws3=to_dev(L["Ws3"]))
    y, _ = moe.moe_grouped_down(h, offs, to_dev(L["W2"]), T, k, Ws2=to_dev(L["Ws2"]))
    torch.cuda.synchronize()
    S = T * k
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(S, size=256, replace=False))
    # include every group boundary row and the last row
    rows = np.unique(np.concatenate([rows, pm["offsets"][1:-1], pm["offsets"][1:-1] - 1, [S - 1]]))
    rows = rows[(rows >= 0) & (rows < S)]
    expert = np.searchsorted(pm["offsets"], rows, side="right") - 1
    h_got = to_f64(h[torch.from_numpy(rows).cuda()])
    y_got = to_f64(y[torch.from_numpy(rows).cuda()])
    for e in np.unique(expert):
        sel = expert == e
        xs = orc.bf16_to_f64(xs_bits[rows[sel]])
        one = np.array([0, int(sel.sum())])
        h_ref = orc.grouped_swiglu(xs, orc.bf16_to_f64(L["W1"][e:e + 1]), orc.bf16_to_f64(L["W3"][e:e + 1]), one)
        assert_close(h_got[sel], h_ref, f"h expert {e}", atol=H_ATOL, rtol=H_RTOL)
        y_ref = orc.grouped_down(h_got[sel], orc.bf16_to_f64(L["W2"][e:e + 1]), one)
        assert_close(y_got[sel], y_ref, f"y expert {e}", atol=H_ATOL, rtol=H_RTOL)
    assert moe.device_error() == 0


def test_bounded_wait_times_out_and_reports(moe):
    """Failure detection without a GPU fault: a wait on a barrier that nothing
    signals gives up after its limit, the status is read on the host, and the
    context stays usable for the next layer call."""
    from grouped_gemm_router_gb300 import _native as N
    import ctypes
    assert moe.device_error() == 0
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = N.lib.moe_selftest_wait_timeout(2000, ctypes.c_void_p(flag.data_ptr()), None)
    assert st == N.MOE_OK
    torch.cuda.synchronize()
    assert int(flag.item()) == 1
    assert moe.device_error() == N.MOE_ERR_DEVICE_TIMEOUT
    assert moe.device_error() == 0          # read-and-clear
    # the context still runs the layer correctly
    w_, L = _layer(256, 128, 256, 4, 2, False, 10)
    ids, w, pm, xs_bits = _grouped_inputs(L, 2, 4)
    h = moe.moe_grouped_swiglu(to_dev(xs_bits), to_dev(pm["offsets"]), to_dev(L["W1"]), to_dev(L["W3"]), 256, 2)
    torch.cuda.synchronize()
    h_ref = orc.grouped_swiglu(orc.bf16_to_f64(xs_bits), orc.bf16_to_f64(L["W1"]), orc.bf16_to_f64(L["W3"]),
                               pm["offsets"])
    assert_close(to_f64(h), h_ref, "h after a timed-out wait", atol=H_ATOL, rtol=H_RTOL)
    assert moe.device_error() == 0
