"""A second, independent statement of the layer, pinned against the oracle.

The dispatch of "Chinchilla scaling, MoE, and fused Triton kernels" (section
"PyTorch MoE implementation") is restated here in plain PyTorch fp64 on the
CPU -- torch.topk, a softmax over the selected logits, a stable argsort of
the flattened ids, bincount, repeat_interleave, one SwiGLU expert per group
and the inverse permutation with the weighted sum -- in code written for this
test, with the SwiGLU activation of "Triton MoE Kernels & Memory
Checkpointing", Part A, section 2.  The numpy oracle must agree to rounding.
Inputs keep every top-k margin away from ties, where torch.topk's order of
equal values is unspecified."""
import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

from grouped_gemm_router_gb300 import inputs
from oracle import moe_oracle as orc


def moe_ffn_torch(x, Wg, W1, W3, W2, k, bias=None, Ws=None):
    T, D = x.shape
    E = W1.shape[0]
    logits = x @ Wg
    if bias is not None:
        logits = logits + bias
    top_v, top_i = torch.topk(logits, k, dim=-1)          # descending
    gate = torch.softmax(top_v, dim=-1)
    flat = top_i.reshape(-1)
    order = torch.argsort(flat, stable=True)
    counts = torch.bincount(flat, minlength=E)
    xs = x.repeat_interleave(k, dim=0)[order]
    ys = torch.zeros_like(xs)
    start = 0
    for e in range(E):
        n = int(counts[e])
        if n:
            rows = xs[start:start + n]
            ys[start:start + n] = (Fn.silu(rows @ W1[e]) * (rows @ W3[e])) @ W2[e]
        start += n
    inv = torch.empty_like(order)
    inv[order] = torch.arange(order.numel())
    out = (gate.unsqueeze(-1) * ys[inv].view(T, k, D)).sum(dim=1)
    if Ws is not None:
        s1, s3, s2 = Ws
        out = out + (Fn.silu(x @ s1) * (x @ s3)) @ s2
    return out, top_i


@pytest.mark.parametrize("T,D,F,E,k,shared,seed", [
    (64, 32, 48, 4, 2, False, 1),
    (50, 16, 24, 6, 3, True, 2),
    (40, 24, 16, 5, 5, True, 3),     # k = E
    (80, 32, 32, 8, 1, False, 4),
])
def test_torch_restatement_matches_oracle(T, D, F, E, k, shared, seed):
    _, L = inputs.make_custom(T, D, F, E, k, shared, seed)
    f64 = {n: orc.bf16_to_f64(L[n]) for n in ("x", "Wg", "W1", "W3", "W2")}
    if shared:
        f64.update({n: orc.bf16_to_f64(L[n]) for n in ("Ws1", "Ws3", "Ws2")})
    gap = orc.topk_gap(orc.router_logits(f64["x"], f64["Wg"]), k)
    assert gap.min() > 1e-9, "inputs with an exact tie: torch.topk's order is unspecified there"
    t = {n: torch.from_numpy(a) for n, a in f64.items()}
    out_t, ids_t = moe_ffn_torch(t["x"], t["Wg"], t["W1"], t["W3"], t["W2"], k,
                                 Ws=(t["Ws1"], t["Ws3"], t["Ws2"]) if shared else None)
    ref = orc.moe_ffn_forward(L["x"], L["Wg"], L["W1"], L["W3"], L["W2"], k, Ws1=L["Ws1"], Ws3=L["Ws3"],
                              Ws2=L["Ws2"], return_all=True)
    assert (ids_t.numpy() == ref["ids"]).all()
    assert np.abs(out_t.numpy() - ref["out"]).max() <= 1e-12 * max(1.0, np.abs(ref["out"]).max())
