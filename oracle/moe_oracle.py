"""Plain fp64 CPU oracle of the mixture-of-experts SwiGLU FFN forward pass.

TEST INFRASTRUCTURE.  Only the tests, the package's smoke check and the
benchmark's CPU-baseline / reference arm may import or run this module.  The
CUDA library never calls it and shares no code with it; it imports nothing
from the package.

What it computes is the layer as the pages define it, step by step, each step
in the order and notation of the pages, with no blocking, fusion or
reordering beyond what the definition states.  Every floating-point value is
carried in float64: the bf16 inputs are widened exactly, and nothing is
rounded back to bf16 along the way.  Library primitives (a matmul, a stable
sort, a bincount) serve as steps where the pages use the same primitive.

Sources (page title, section):
  [P1] "Triton MoE Kernels & Memory Checkpointing" -- Part A, sections 2
       ("Why it matters here": SwiGLU expert W2(silu(W1 x) * W3 x), top-2 of 8
       routed experts plus a shared expert, the W1/W3 FLOP count), 6.2, 10.2
       (the per-expert reference loop that skips empty experts) and 10.3 (the
       sort-by-expert dispatch layout).
  [P3] "Chinchilla scaling, MoE, and fused Triton kernels" -- section
       "PyTorch MoE implementation" (router logits x @ gate_w, top-k, softmax
       over the selected logits, stable argsort of the flattened ids, bincount,
       gather, grouped GEMMs, inverse permutation and weighted sum).

Readings where the pages are silent or contradict one another:
  * Activation: the P3 listing applies silu to one up-projection and then
    multiplies by itself; its fused kernel applies plain silu.  Both disagree
    with the SwiGLU expert of P1 section 2 and section 8.  The oracle follows
    SwiGLU: h = silu(x W1) * (x W3).
  * Weight orientation: P1 stores nn.Linear weights [E, F, D]; P3 stores
    [E, D, F] and [E, F, D] and multiplies x @ W.  The oracle follows P3.
  * Top-k order and ties: descending logits (torch.topk order), equal logits
    resolved toward the lower expert index.
  * Softmax is over the k selected logits, after top-k (P3 listing).
  * Stable permutation: within one expert, slots keep ascending slot order
    s = t*k + j (stable argsort of the row-major flattened ids).
  * Shared expert: an always-on SwiGLU expert of the same shape, added to every
    token's output with weight 1.
  * Router bias: an optional fp32 [E] vector added to the logits (used to
    impose a skewed expert load); zero when absent.
"""
from __future__ import annotations

import numpy as np


# ----------------------------------------------------------------------------
# bf16 widening (exact)
# ----------------------------------------------------------------------------
def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float64.  A bf16 value is the top
    16 bits of the float32 with the same sign, exponent and leading mantissa
    bits, so the widening is exact."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# Step 1: router logits                                  [P3 PyTorch MoE]
# ----------------------------------------------------------------------------
def router_logits(x: np.ndarray, Wg: np.ndarray, bias: np.ndarray | None = None) -> np.ndarray:
    """logits[t, e] = sum_d x[t, d] * Wg[d, e]  (+ bias[e]).   x [T,D], Wg [D,E]."""
    logits = x @ Wg
    if bias is not None:
        logits = logits + np.asarray(bias, dtype=np.float64)[None, :]
    return logits


# ----------------------------------------------------------------------------
# Step 2: top-k selection, softmax over the selected logits  [P3 PyTorch MoE]
# ----------------------------------------------------------------------------
def topk_softmax(logits: np.ndarray, k: int) -> tuple[np.ndarray, np.ndarray]:
    """ids[t, :] = the k largest logits of row t, in descending order, equal
    logits taken in ascending expert order; w[t, :] = softmax of those k
    logits.  Returns (ids int32 [T,k], w float64 [T,k])."""
    T, E = logits.shape
    if not 1 <= k <= E:
        raise ValueError("k must satisfy 1 <= k <= E")
    # A stable sort of the negated logits lists equal logits by expert index.
    order = np.argsort(-logits, axis=1, kind="stable")
    ids = order[:, :k].astype(np.int32)
    sel = np.take_along_axis(logits, order[:, :k], axis=1)
    z = np.exp(sel - sel[:, :1])          # sel[:, 0] is the largest selected logit
    w = z / z.sum(axis=1, keepdims=True)
    return ids, w


def topk_gap(logits: np.ndarray, k: int) -> np.ndarray:
    """Margin between the k-th and (k+1)-th largest logit of each token (inf
    when k == E).  A token with a small margin can legitimately select a
    different expert set under a different summation order."""
    T, E = logits.shape
    if k == E:
        return np.full(T, np.inf)
    s = -np.sort(-logits, axis=1)
    return s[:, k - 1] - s[:, k]


# ----------------------------------------------------------------------------
# Step 3: flatten, stable sort by expert, counts, offsets, inverse
#                                          [P3 PyTorch MoE; P1 10.3 steps 1-2]
# ----------------------------------------------------------------------------
def permutation(ids: np.ndarray, E: int) -> dict:
    """Slots s = t*k + j are the row-major flattening of ids [T,k].
    perm[p] = the slot at sorted position p (stable argsort by expert id),
    counts[e] = number of slots routed to e, offsets = exclusive prefix sum of
    counts with offsets[E] = T*k, inv[perm[p]] = p."""
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    perm = np.argsort(flat, kind="stable")
    counts = np.bincount(flat, minlength=E)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size)
    return {
        "perm": perm.astype(np.int32),
        "inv": inv.astype(np.int32),
        "counts": counts.astype(np.int32),
        "offsets": offsets.astype(np.int32),
    }


def gather_sorted(x: np.ndarray, perm: np.ndarray, k: int) -> np.ndarray:
    """x_sorted = x.repeat_interleave(k, 0)[perm]: row p is token perm[p] // k."""
    return x[np.asarray(perm, dtype=np.int64) // k]


# ----------------------------------------------------------------------------
# Step 4: expert SwiGLU up-projection per expert       [P1 sections 2, 10.2]
# ----------------------------------------------------------------------------
def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z * sigmoid(z) = z / (1 + exp(-z)), sigmoid the logistic function."""
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def grouped_swiglu(x_sorted: np.ndarray, W1: np.ndarray, W3: np.ndarray,
                   offsets: np.ndarray) -> np.ndarray:
    """h[p] = silu(x_sorted[p] @ W1[e]) * (x_sorted[p] @ W3[e]) for every
    sorted position p of expert e.  Empty experts are skipped; every row of h
    belongs to exactly one expert.  W1, W3 [E, D, F]."""
    E = W1.shape[0]
    S = x_sorted.shape[0]
    h = np.zeros((S, W1.shape[2]), dtype=np.float64)
    for e in range(E):
        start, end = int(offsets[e]), int(offsets[e + 1])
        if end == start:
            continue
        chunk = x_sorted[start:end]
        g = chunk @ W1[e]
        u = chunk @ W3[e]
        h[start:end] = silu(g) * u
    return h


# ----------------------------------------------------------------------------
# Step 5: expert down-projection per expert          [P1 10.3 step 4; P3]
# ----------------------------------------------------------------------------
def grouped_down(h: np.ndarray, W2: np.ndarray, offsets: np.ndarray) -> np.ndarray:
    """y[p] = h[p] @ W2[e] for every sorted position p of expert e.  W2 [E,F,D]."""
    E = W2.shape[0]
    y = np.zeros((h.shape[0], W2.shape[2]), dtype=np.float64)
    for e in range(E):
        start, end = int(offsets[e]), int(offsets[e + 1])
        if end == start:
            continue
        y[start:end] = h[start:end] @ W2[e]
    return y


# ----------------------------------------------------------------------------
# Shared expert: always on, unweighted                        [P1 section 2]
# ----------------------------------------------------------------------------
def shared_expert(x: np.ndarray, Ws1: np.ndarray, Ws3: np.ndarray, Ws2: np.ndarray) -> np.ndarray:
    """ys[t] = (silu(x[t] @ Ws1) * (x[t] @ Ws3)) @ Ws2."""
    return (silu(x @ Ws1) * (x @ Ws3)) @ Ws2


# ----------------------------------------------------------------------------
# Step 6: un-permute and weighted combine                 [P3 PyTorch MoE]
# ----------------------------------------------------------------------------
def combine(y_sorted: np.ndarray, inv: np.ndarray, w: np.ndarray,
            ys: np.ndarray | None = None) -> np.ndarray:
    """out[t] = sum_j w[t, j] * y_sorted[inv[t*k + j]]  (+ ys[t])."""
    T, k = w.shape
    y_tok = y_sorted[np.asarray(inv, dtype=np.int64)].reshape(T, k, -1)
    out = (w[:, :, None] * y_tok).sum(axis=1)
    if ys is not None:
        out = out + ys
    return out


# ----------------------------------------------------------------------------
# The whole layer
# ----------------------------------------------------------------------------
def moe_ffn_forward(x, Wg, W1, W3, W2, k, bias=None, Ws1=None, Ws3=None, Ws2=None,
                    ids=None, weights=None, return_all=False):
    """Forward pass of one MoE SwiGLU FFN layer in float64.

    Array arguments are bf16 bit patterns (uint16) or float64 arrays; `bias`
    is fp32/fp64 [E] or None; the shared expert is present when Ws1, Ws3 and
    Ws2 are all given.  `ids`/`weights` ([T,k]) replace steps 1-2 when given
    (routing fixed from outside)."""
    f = lambda a: a if (a is None or a.dtype == np.float64) else bf16_to_f64(a)
    x, Wg, W1, W3, W2 = f(x), f(Wg), f(W1), f(W3), f(W2)
    E = W1.shape[0]
    logits = router_logits(x, Wg, bias)
    if ids is None:
        ids, w = topk_softmax(logits, k)
    else:
        ids = np.asarray(ids, dtype=np.int32)
        w = np.asarray(weights, dtype=np.float64)
    pm = permutation(ids, E)
    xs = gather_sorted(x, pm["perm"], k)
    h = grouped_swiglu(xs, W1, W3, pm["offsets"])
    y = grouped_down(h, W2, pm["offsets"])
    ys = None
    if Ws1 is not None:
        ys = shared_expert(x, f(Ws1), f(Ws3), f(Ws2))
    out = combine(y, pm["inv"], w, ys)
    if not return_all:
        return out
    return dict(out=out, logits=logits, ids=ids, w=w, h=h, y=y, ys=ys, **pm)


# ----------------------------------------------------------------------------
# FLOP accounting                                         [P1 section 2]
# ----------------------------------------------------------------------------
def w1w3_flops(T: int, D: int, F: int, k: int) -> int:
    """FLOPs of the routed W1 and W3 GEMMs: each of the T*k routed slots does
    two [D] x [D,F] products at 2 FLOPs per multiply-add."""
    return 2 * (2 * T * k * D * F)


def active_flops(T: int, D: int, F: int, E: int, k: int, shared: bool) -> int:
    """Router GEMM + routed W1/W3/W2 + (optional) shared-expert W1/W3/W2."""
    return 2 * T * D * E + 3 * (2 * T * k * D * F) + (3 * (2 * T * D * F) if shared else 0)
