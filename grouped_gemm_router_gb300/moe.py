"""PyTorch-facing entry points of the MoE SwiGLU FFN forward pass.

These functions only allocate outputs with torch, check shapes/dtypes, and
call the C ABI of libmoeffn.so on the current CUDA stream.  Tensor layouts:
  x [T, D] bf16, Wg [D, E] bf16, bias [E] fp32 (optional),
  W1, W3 [E, D, F] bf16, W2 [E, F, D] bf16,
  shared expert Ws1, Ws3 [D, F], Ws2 [F, D] bf16 (optional).
"""
from __future__ import annotations

import ctypes

import torch

from . import _native as N
from ._native import check, lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _need(t, name, dtype, shape=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def layer_dims(x, W1, k):
    T, D = x.shape
    E, _, F = W1.shape
    return T, D, F, E, k


def workspace_size(T, D, F, E, k, shared, host_io=False) -> int:
    n = lib.moe_ffn_workspace_size(N.dims(T, D, F, E, k), int(bool(shared)), int(bool(host_io)))
    if n == 0:
        raise N.MoeError(N.MOE_ERR_UNSUPPORTED_SHAPE, "moe_ffn_workspace_size")
    return n


class Workspace:
    """Device workspace of moe_ffn_forward, with typed views of its regions
    (the layout documented in moe_ffn.h)."""

    def __init__(self, T, D, F, E, k, shared, host_io=False, device=None):
        self.dims = (T, D, F, E, k)
        self.shared = bool(shared)
        self.nbytes = workspace_size(T, D, F, E, k, shared, host_io)
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device or "cuda")

    def views(self):
        T, D, F, E, k = self.dims
        S = T * k
        rows = S + (T if self.shared else 0)
        nblk = N.route_blocks(T)           # rows in use on this device
        nblk_max = (T + 15) // 16           # rows reserved (16-token blocks)
        out, off = {}, 0

        def take(name, n, dtype, shape):
            nonlocal off
            size = n * torch.tensor([], dtype=dtype).element_size()
            out[name] = self.buf[off:off + size].view(dtype).view(*shape)
            off += (size + 255) // 256 * 256

        npack = int(lib.moe_route_scratch_size(N.dims(T, D, F, E, k)))
        take("router_packed", npack, torch.uint8, (npack,))
        take("ids", S, torch.int32, (T, k))
        take("w", S, torch.float32, (T, k))
        take("hist", nblk_max * E, torch.int32, (nblk_max, E))
        out["hist"] = out["hist"][:nblk]
        take("counts", E, torch.int32, (E,))
        take("offsets", E + 1, torch.int32, (E + 1,))
        take("perm", S, torch.int32, (S,))
        take("inv", S, torch.int32, (S,))
        take("x_sorted", S * D, torch.bfloat16, (S, D))
        take("h", rows * F, torch.bfloat16, (rows, F))
        take("y", S * D, torch.bfloat16, (S, D))
        if self.shared:
            take("ys", T * D, torch.float32, (T, D))
        return out


def _options(stage_events=None, ids_in=None, weights_in=None, chained=False):
    if stage_events is None and ids_in is None and not chained:
        return None
    o = N.MoeOptions()
    o.flags = N.MOE_FFN_CHAINED if chained else 0
    for i, ev in enumerate(stage_events or []):
        if ev is None:
            continue
        handle = ev.cuda_event if hasattr(ev, "cuda_event") else int(ev)
        if not handle:
            # torch creates the CUDA event lazily, on its first record()
            ev.record()
            handle = ev.cuda_event
        o.stage_events[i] = handle
    if ids_in is not None:
        _need(ids_in, "ids_in", torch.int32)
        _need(weights_in, "weights_in", torch.float32)
        o.ids_in = ids_in.data_ptr()
        o.weights_in = weights_in.data_ptr()
    return ctypes.byref(o)


def moe_ffn_forward(x, Wg, W1, W3, W2, k, bias=None, Ws1=None, Ws3=None, Ws2=None, out=None,
                    workspace: Workspace | None = None, stage_events=None, ids_in=None,
                    weights_in=None, chained=False):
    """Forward pass of the MoE SwiGLU FFN layer; returns out [T, D] bf16.
    chained=True runs W1||W3 and W2 as one kernel with h kept on chip
    (D <= 256)."""
    T, D, F, E, k = layer_dims(x, W1, k)
    shared = Ws1 is not None
    for t, n, shp in ((x, "x", (T, D)), (Wg, "Wg", (D, E)), (W1, "W1", (E, D, F)),
                      (W3, "W3", (E, D, F)), (W2, "W2", (E, F, D)), (Ws1, "Ws1", (D, F)),
                      (Ws3, "Ws3", (D, F)), (Ws2, "Ws2", (F, D))):
        _need(t, n, torch.bfloat16, shp)
    _need(bias, "bias", torch.float32, (E,))
    if out is None:
        out = torch.empty(T, D, dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = Workspace(T, D, F, E, k, shared, device=x.device)
    st = lib.moe_ffn_forward(_ptr(x), _ptr(Wg), _ptr(bias), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(Ws1),
                             _ptr(Ws3), _ptr(Ws2), N.dims(T, D, F, E, k), _ptr(out),
                             _ptr(workspace.buf), workspace.nbytes,
                             _options(stage_events, ids_in, weights_in, chained), _stream())
    check(st, "moe_ffn_forward")
    return out


def moe_ffn_forward_host(x_host, Wg, W1, W3, W2, k, out_host, workspace: Workspace, bias=None,
                         Ws1=None, Ws3=None, Ws2=None, stage_events=None):
    """Forward pass with x and out in (pinned) host memory; copies are part of
    the call, enqueued on the current stream."""
    T, D, F, E, k = layer_dims(x_host, W1, k)
    if x_host.is_cuda or out_host.is_cuda:
        raise ValueError("x_host and out_host must be host tensors")
    st = lib.moe_ffn_forward_host(_ptr(x_host), _ptr(Wg), _ptr(bias), _ptr(W1), _ptr(W3), _ptr(W2),
                                  _ptr(Ws1), _ptr(Ws3), _ptr(Ws2), N.dims(T, D, F, E, k),
                                  _ptr(out_host), _ptr(workspace.buf), workspace.nbytes,
                                  _options(stage_events), _stream())
    check(st, "moe_ffn_forward_host")
    return out_host


class BackwardWorkspace:
    """Device workspace of moe_ffn_backward, with typed views of its regions
    (the layout documented in moe_ffn.h: padded sorted rows, the shared rows
    from S_pad = T*k + 64*E)."""

    def __init__(self, T, D, F, E, k, shared, device=None):
        self.dims = (T, D, F, E, k)
        self.shared = bool(shared)
        self.nbytes = int(lib.moe_ffn_backward_workspace_size(N.dims(T, D, F, E, k), int(bool(shared))))
        if self.nbytes == 0 and T > 0:
            raise N.MoeError(N.MOE_ERR_UNSUPPORTED_SHAPE, "moe_ffn_backward_workspace_size")
        self.buf = torch.empty(max(self.nbytes, 256), dtype=torch.uint8, device=device or "cuda")

    def views(self):
        T, D, F, E, k = self.dims
        S = T * k
        Sp = S + 64 * E
        rows = Sp + (T if self.shared else 0)
        out, off = {"S_pad": Sp}, 0

        def take(name, n, dtype, shape):
            nonlocal off
            size = n * torch.tensor([], dtype=dtype).element_size()
            out[name] = self.buf[off:off + size].view(dtype).view(*shape)
            off += (size + 255) // 256 * 256

        take("ybar", Sp * D, torch.bfloat16, (Sp, D))
        take("hbar", rows * F, torch.bfloat16, (rows, F))
        take("gu", rows * 2 * F, torch.bfloat16, (rows, 2 * F))
        take("h", rows * F, torch.bfloat16, (rows, F))
        take("xbar", rows * D, torch.bfloat16, (rows, D))
        take("wbar", S, torch.float32, (T, k))
        take("lbar", S, torch.float32, (T, k))
        return out


def padded_rows(counts):
    """Row of each sorted position in the backward's padded layout: group e
    starts at the sum of the earlier group sizes rounded up to 64."""
    counts = [int(c) for c in counts]
    prow0, run = [], 0
    for c in counts:
        prow0.append(run)
        run += (c + 63) // 64 * 64
    idx = []
    for e, c in enumerate(counts):
        idx.extend(range(prow0[e], prow0[e] + c))
    return idx


def moe_ffn_backward(x, Wg, W1, W3, W2, k, d_out, workspace: Workspace, Ws1=None, Ws3=None, Ws2=None,
                     bwd_workspace: BackwardWorkspace | None = None, ids_in=None, weights_in=None,
                     router=True, stage_events=None, chained=False):
    """Gradients of sum(d_out * out) for the forward call that filled
    `workspace`.  Returns dict(dx bf16 [T, D], dW1, dW3 [E, D, F], dW2 [E, F, D]
    (+ dWs1, dWs3, dWs2), and with router=True dWg [D, E], dbias [E]) fp32.
    chained: the forward call ran with chained=True (its workspace has no h)."""
    T, D, F, E, k = layer_dims(x, W1, k)
    shared = Ws1 is not None
    _need(d_out, "d_out", torch.bfloat16, (T, D))
    dev = x.device
    f32 = dict(dtype=torch.float32, device=dev)
    g = dict(dx=torch.empty(T, D, dtype=torch.bfloat16, device=dev),
             dW1=torch.empty(E, D, F, **f32), dW3=torch.empty(E, D, F, **f32), dW2=torch.empty(E, F, D, **f32))
    if shared:
        g.update(dWs1=torch.empty(D, F, **f32), dWs3=torch.empty(D, F, **f32), dWs2=torch.empty(F, D, **f32))
    if router:
        g.update(dWg=torch.empty(D, E, **f32), dbias=torch.empty(E, **f32))
    if bwd_workspace is None:
        bwd_workspace = BackwardWorkspace(T, D, F, E, k, shared, device=dev)
    st = lib.moe_ffn_backward(_ptr(x), _ptr(Wg), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(Ws1), _ptr(Ws3), _ptr(Ws2),
                              _ptr(d_out), N.dims(T, D, F, E, k), _ptr(workspace.buf), workspace.nbytes,
                              _ptr(g["dx"]), _ptr(g.get("dWg")), _ptr(g.get("dbias")), _ptr(g["dW1"]),
                              _ptr(g["dW3"]), _ptr(g["dW2"]), _ptr(g.get("dWs1")), _ptr(g.get("dWs3")),
                              _ptr(g.get("dWs2")), _ptr(bwd_workspace.buf), bwd_workspace.nbytes,
                              _options(stage_events, ids_in, weights_in, chained), _stream())
    check(st, "moe_ffn_backward")
    return g


def moe_route(x, Wg, k, bias=None):
    """Router GEMM + top-k + softmax -> (ids [T,k] int32, weights [T,k] fp32,
    block_hist [ceil(T/TB), E] int32 with TB = moe_route_block_tokens(T))."""
    T, D = x.shape
    E = Wg.shape[1]
    _need(x, "x", torch.bfloat16, (T, D))
    _need(Wg, "Wg", torch.bfloat16, (D, E))
    _need(bias, "bias", torch.float32, (E,))
    ids = torch.empty(T, k, dtype=torch.int32, device=x.device)
    w = torch.empty(T, k, dtype=torch.float32, device=x.device)
    hist = torch.empty(N.route_blocks(T), E, dtype=torch.int32, device=x.device)
    d = N.dims(T, D, 64, E, k)
    nscratch = int(lib.moe_route_scratch_size(d))
    scratch = torch.empty(max(nscratch, 16), dtype=torch.uint8, device=x.device)
    st = lib.moe_route(_ptr(x), _ptr(Wg), _ptr(bias), d, _ptr(ids), _ptr(w), _ptr(hist), _ptr(scratch),
                       nscratch, _stream())
    check(st, "moe_route")
    return ids, w, hist


def moe_permute(ids, E, x=None):
    """Stable expert-grouped permutation of ids [T, k]; with x, also the
    gathered x_sorted [T*k, D]."""
    T, k = ids.shape
    _need(ids, "ids", torch.int32, (T, k))
    D = x.shape[1] if x is not None else 64
    if x is not None:
        _need(x, "x", torch.bfloat16, (T, D))
    d = N.dims(T, D, 64, E, k)
    dev = ids.device
    S = T * k
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(S, dtype=torch.int32, device=dev)
    inv = torch.empty(S, dtype=torch.int32, device=dev)
    xs = torch.empty(S, D, dtype=torch.bfloat16, device=dev) if x is not None else None
    nscratch = max(int(lib.moe_permute_scratch_size(d)), 16)
    scratch = torch.empty(nscratch, dtype=torch.uint8, device=dev)
    st = lib.moe_permute(_ptr(ids), d, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv), _ptr(x),
                         _ptr(xs), _ptr(scratch), nscratch, _stream())
    check(st, "moe_permute")
    return dict(counts=counts, offsets=offsets, perm=perm, inv=inv, x_sorted=xs)


def moe_grouped_swiglu(x_sorted, offsets, W1, W3, T, k, x=None, Ws1=None, Ws3=None, h=None):
    """h [T*k (+T), F] = silu(A W1[e]) * (A W3[e]) per expert group (+ shared rows)."""
    S, D = x_sorted.shape
    E, _, F = W1.shape
    shared = Ws1 is not None
    _need(x_sorted, "x_sorted", torch.bfloat16, (T * k, D))
    _need(W1, "W1", torch.bfloat16, (E, D, F))
    _need(W3, "W3", torch.bfloat16, (E, D, F))
    _need(offsets, "offsets", torch.int32, (E + 1,))
    if shared:
        _need(x, "x", torch.bfloat16, (T, D))
        _need(Ws1, "Ws1", torch.bfloat16, (D, F))
        _need(Ws3, "Ws3", torch.bfloat16, (D, F))
    rows = T * k + (T if shared else 0)
    if h is None:
        h = torch.empty(rows, F, dtype=torch.bfloat16, device=x_sorted.device)
    st = lib.moe_grouped_swiglu(_ptr(x_sorted), _ptr(x), _ptr(W1), _ptr(W3), _ptr(Ws1), _ptr(Ws3),
                                _ptr(offsets), N.dims(T, D, F, E, k), _ptr(h), _stream())
    check(st, "moe_grouped_swiglu")
    return h


def moe_grouped_down(h, offsets, W2, T, k, Ws2=None, y=None, ys=None):
    """(y [T*k, D] bf16, ys [T, D] fp32 or None): y = h W2[e] per expert
    group; with Ws2, ys = the shared rows of h times Ws2."""
    E, F, D = W2.shape
    shared = Ws2 is not None
    rows = T * k + (T if shared else 0)
    _need(h, "h", torch.bfloat16, (rows, F))
    _need(W2, "W2", torch.bfloat16, (E, F, D))
    _need(Ws2, "Ws2", torch.bfloat16, (F, D))
    _need(offsets, "offsets", torch.int32, (E + 1,))
    if y is None:
        y = torch.empty(T * k, D, dtype=torch.bfloat16, device=h.device)
    if shared and ys is None:
        ys = torch.empty(T, D, dtype=torch.float32, device=h.device)
    _need(y, "y", torch.bfloat16, (T * k, D))
    if shared:
        _need(ys, "ys", torch.float32, (T, D))
    st = lib.moe_grouped_down(_ptr(h), _ptr(W2), _ptr(Ws2), _ptr(offsets), N.dims(T, D, F, E, k),
                              _ptr(y), _ptr(ys if shared else None), _stream())
    check(st, "moe_grouped_down")
    return y, (ys if shared else None)


def moe_grouped_ffn_chained(x_sorted, offsets, W1, W3, W2, T, k, x=None, Ws1=None, Ws3=None,
                            Ws2=None, y=None, ys=None):
    """(y [T*k, D] bf16, ys [T, D] fp32 or None) = (silu(A W1[e]) * (A W3[e]))
    W2[e] per expert group (+ the shared expert's rows), in one kernel that
    never writes h (D <= 256)."""
    S, D = x_sorted.shape
    E, _, F = W1.shape
    shared = Ws1 is not None
    _need(x_sorted, "x_sorted", torch.bfloat16, (T * k, D))
    _need(W1, "W1", torch.bfloat16, (E, D, F))
    _need(W3, "W3", torch.bfloat16, (E, D, F))
    _need(W2, "W2", torch.bfloat16, (E, F, D))
    _need(offsets, "offsets", torch.int32, (E + 1,))
    if shared:
        _need(x, "x", torch.bfloat16, (T, D))
        _need(Ws1, "Ws1", torch.bfloat16, (D, F))
        _need(Ws3, "Ws3", torch.bfloat16, (D, F))
        _need(Ws2, "Ws2", torch.bfloat16, (F, D))
    if y is None:
        y = torch.empty(T * k, D, dtype=torch.bfloat16, device=x_sorted.device)
    if shared and ys is None:
        ys = torch.empty(T, D, dtype=torch.float32, device=x_sorted.device)
    _need(y, "y", torch.bfloat16, (T * k, D))
    if shared:
        _need(ys, "ys", torch.float32, (T, D))
    st = lib.moe_grouped_ffn_chained(_ptr(x_sorted), _ptr(x), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(Ws1),
                                     _ptr(Ws3), _ptr(Ws2), _ptr(offsets), N.dims(T, D, F, E, k), _ptr(y),
                                     _ptr(ys if shared else None), _stream())
    check(st, "moe_grouped_ffn_chained")
    return y, (ys if shared else None)


def moe_combine(y, weights, inv, ys=None, out=None):
    """out[t] = sum_j weights[t, j] * y[inv[t*k + j]] (+ ys[t], fp32)."""
    T, k = weights.shape
    D = y.shape[1]
    _need(y, "y", torch.bfloat16, (T * k, D))
    _need(ys, "ys", torch.float32, (T, D))
    _need(weights, "weights", torch.float32, (T, k))
    _need(inv, "inv", torch.int32, (T * k,))
    if out is None:
        out = torch.empty(T, D, dtype=torch.bfloat16, device=y.device)
    E = max(k, 1)
    st = lib.moe_combine(_ptr(y), _ptr(ys), _ptr(weights), _ptr(inv), N.dims(T, D, 64, E, k),
                         _ptr(out), _stream())
    check(st, "moe_combine")
    return out


def device_error() -> int:
    return int(lib.moe_device_error())


def launch_count() -> int:
    return int(lib.moe_launch_count())
