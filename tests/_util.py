"""Helpers shared by the tests: bf16 bit arrays <-> torch tensors, tolerance."""
import numpy as np
import torch

RTOL = 1e-2   # |gpu - oracle| <= ATOL + RTOL * |oracle|, elementwise
ATOL = 1e-2


def to_dev(a, device="cuda"):
    """numpy uint16 bf16 bits (or float32/int32 arrays) -> CUDA tensor."""
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(a).to(device)


def bf16_bits(t):
    """bf16 CUDA tensor -> numpy uint16 bits."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def within_tol(got, ref, atol=ATOL, rtol=RTOL):
    """Returns (ok, n_bad, max_abs_diff, worst excess)."""
    diff = np.abs(got - ref)
    excess = diff - (atol + rtol * np.abs(ref))
    return bool((excess <= 0).all()), int((excess > 0).sum()), float(diff.max(initial=0.0)), float(excess.max(initial=-1.0))


def assert_close(got, ref, what, atol=ATOL, rtol=RTOL):
    ok, nbad, mx, ex = within_tol(got, ref, atol, rtol)
    assert ok, f"{what}: {nbad} of {got.size} elements outside {atol} + {rtol}|ref| (max |diff| {mx:.3e})"
    return mx
