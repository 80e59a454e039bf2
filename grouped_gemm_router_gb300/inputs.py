"""Seeded synthetic inputs for the MoE SwiGLU FFN layer.

This module is shared by the CUDA path's tests/benchmark and by the oracle's
tests.  It holds no arithmetic of the layer itself: it only draws normal
numbers, scales them by the stated init, rounds them to bf16, and (for the
skewed-load workload) builds a fixed router bias.

Layouts follow the PyTorch MoE listing on "Chinchilla scaling, MoE, and fused
Triton kernels" (section "PyTorch MoE implementation"):
  x  [T, D]      Wg [D, E]      W1, W3 [E, D, F]      W2 [E, F, D]
and the optional shared expert Ws1, Ws3 [D, F], Ws2 [F, D].

bf16 tensors are carried as numpy uint16 bit patterns (round-to-nearest-even
from float32), so that both sides see the same bytes.

Random numbers: numpy PCG64 seeded with the workload's seed, standard normals
drawn in float32, in the fixed order x, Wg, W1, W3, W2, Ws1, Ws3, Ws2.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    D: int
    F: int
    E: int
    k: int
    shared: bool
    seed: int
    zipf_s: float | None = None      # skewed router load (Zipf exponent)
    empty_expert: int | None = None  # expert forced to receive no tokens

    @property
    def S(self) -> int:
        return self.T * self.k


# The five synthetic workloads of the MoE FFN forward.
WORKLOADS = {
    "tiny": Workload("tiny", T=256, D=128, F=256, E=4, k=2, shared=False, seed=0),
    "gptoss_lite": Workload("gptoss_lite", T=32768, D=768, F=1536, E=8, k=2,
                            shared=True, seed=1),
    "skewed": Workload("skewed", T=32768, D=768, F=1536, E=8, k=2, shared=False,
                       seed=2, zipf_s=1.2, empty_expert=7),
    "small_chunk": Workload("small_chunk", T=2048, D=768, F=1536, E=64, k=4,
                            shared=True, seed=3),
    "wide": Workload("wide", T=16384, D=2048, F=8192, E=16, k=2, shared=False, seed=4),
}
WORKLOAD_ORDER = ["tiny", "gptoss_lite", "skewed", "small_chunk", "wide"]


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even) and return the uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounded = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(gen: np.random.Generator, shape, std: float) -> np.ndarray:
    a = gen.standard_normal(int(np.prod(shape)), dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return f32_to_bf16_bits(a).reshape(shape)


def zipf_router_bias(E: int, s: float, empty_expert: int | None) -> np.ndarray:
    """Per-expert fp32 logit bias: bias[e] = ln p_e with p_e proportional to
    (e+1)^-s over the experts that may receive tokens, and -1e4 for the expert
    that must stay empty."""
    live = [e for e in range(E) if e != empty_expert]
    p = np.array([(i + 1) ** (-s) for i in range(len(live))], dtype=np.float64)
    p /= p.sum()
    bias = np.zeros(E, dtype=np.float32)
    for i, e in enumerate(live):
        bias[e] = np.float32(math.log(p[i]))
    if empty_expert is not None:
        bias[empty_expert] = np.float32(-1e4)
    return bias


def make_layer(w: Workload) -> dict:
    """Draw one layer's inputs.  Returns a dict of numpy arrays:
    x, Wg, W1, W3, W2 (uint16 bf16 bits), bias (float32 [E] or None),
    Ws1, Ws3, Ws2 (uint16 or None)."""
    T = w.T
    gen = np.random.Generator(np.random.PCG64(w.seed))
    D, F, E = w.D, w.F, w.E
    out = {}
    out["x"] = _normal_bf16(gen, (T, D), 1.0)
    out["Wg"] = _normal_bf16(gen, (D, E), 1.0 / math.sqrt(D))
    out["W1"] = _normal_bf16(gen, (E, D, F), 1.0 / math.sqrt(D))
    out["W3"] = _normal_bf16(gen, (E, D, F), 1.0 / math.sqrt(D))
    out["W2"] = _normal_bf16(gen, (E, F, D), 1.0 / math.sqrt(F))
    if w.shared:
        out["Ws1"] = _normal_bf16(gen, (D, F), 1.0 / math.sqrt(D))
        out["Ws3"] = _normal_bf16(gen, (D, F), 1.0 / math.sqrt(D))
        out["Ws2"] = _normal_bf16(gen, (F, D), 1.0 / math.sqrt(F))
    else:
        out["Ws1"] = out["Ws3"] = out["Ws2"] = None
    out["bias"] = (zipf_router_bias(E, w.zipf_s, w.empty_expert)
                   if w.zipf_s is not None else None)
    return out


def make_custom(T: int, D: int, F: int, E: int, k: int, shared: bool, seed: int,
                bias: np.ndarray | None = None) -> tuple[Workload, dict]:
    """A workload of arbitrary shape with the standard init (for edge cases)."""
    w = Workload(f"custom_T{T}_D{D}_F{F}_E{E}_k{k}", T, D, F, E, k, shared, seed)
    layer = make_layer(w)
    if bias is not None:
        layer["bias"] = np.asarray(bias, dtype=np.float32)
    return w, layer
