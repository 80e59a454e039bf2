"""ctypes binding of libmoeffn.so (argument marshalling only).

Every computation happens in the CUDA library; this module checks tensor
properties, passes raw pointers and the current CUDA stream, and turns status
codes into exceptions.  There is no fallback: if the library is missing or
fails to load, importing the package raises.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoeffn.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED_SHAPE = -2
MOE_ERR_CUDA = -3
MOE_ERR_WORKSPACE = -4
MOE_ERR_DEVICE_TIMEOUT = -5

MOE_FFN_CHAINED = 1
CHAINED_MAX_D = 256

MAX_EXPERTS = 128
MAX_TOPK = 16
MAX_DIM = 8192


class MoeDims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("D", ctypes.c_int32), ("F", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32)]


class MoeOptions(ctypes.Structure):
    _fields_ = [("stage_events", ctypes.c_void_p * 12),
                ("ids_in", ctypes.c_void_p),
                ("weights_in", ctypes.c_void_p),
                ("flags", ctypes.c_uint32)]


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_str(status)} ({status})")


_vp, _sz, _i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int

_SIGNATURES = {
    "moe_ffn_workspace_size": (_sz, [MoeDims, _i32, _i32]),
    "moe_ffn_forward": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, MoeDims, _vp, _vp, _sz,
                               ctypes.POINTER(MoeOptions), _vp]),
    "moe_ffn_forward_host": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, MoeDims, _vp, _vp,
                                    _sz, ctypes.POINTER(MoeOptions), _vp]),
    "moe_ffn_backward_workspace_size": (_sz, [MoeDims, _i32]),
    "moe_ffn_backward": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, MoeDims, _vp, _sz, _vp, _vp, _vp,
                                _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, ctypes.POINTER(MoeOptions), _vp]),
    "moe_route_scratch_size": (_sz, [MoeDims]),
    "moe_route": (_i32, [_vp, _vp, _vp, MoeDims, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_route_block_tokens": (_i32, [_i32]),
    "moe_permute_scratch_size": (_sz, [MoeDims]),
    "moe_permute": (_i32, [_vp, MoeDims, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_grouped_swiglu": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, MoeDims, _vp, _vp]),
    "moe_grouped_down": (_i32, [_vp, _vp, _vp, _vp, MoeDims, _vp, _vp, _vp]),
    "moe_grouped_ffn_chained": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, MoeDims, _vp, _vp, _vp]),
    "moe_combine": (_i32, [_vp, _vp, _vp, _vp, MoeDims, _vp, _vp]),
    "moe_permute_noalloc": (_i32, [_vp, MoeDims, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "moe_device_error": (_i32, []),
    "moe_selftest_wait_timeout": (_i32, [_i32, _vp, _vp]),
    "moe_launch_count": (ctypes.c_uint64, []),
    "moe_status_str": (ctypes.c_char_p, [_i32]),
}


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
            "(the MoE FFN has no CPU fallback)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = load()


def status_str(status: int) -> str:
    return lib.moe_status_str(status).decode()


def check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoeError(status, where)


def dims(T: int, D: int, F: int, E: int, k: int) -> MoeDims:
    return MoeDims(T, D, F, E, k)


def route_blocks(T: int) -> int:
    """Blocks of the router / permutation kernels (rows of the block histogram)."""
    tb = int(lib.moe_route_block_tokens(T))
    return (T + tb - 1) // tb
