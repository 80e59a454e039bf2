"""GB300-native (sm_103a) forward pass of the mixture-of-experts SwiGLU FFN.

The compute path is libmoeffn.so (hand-written CUDA kernels behind a C ABI,
declared in include/moe_ffn.h); `grouped_gemm_router_gb300.moe` is its thin
PyTorch-facing binding.  Importing `moe` loads the library and raises if it
is missing -- there is no CPU fallback.  `inputs` (seeded synthetic inputs)
does not need the library.
"""

__all__ = ["moe", "inputs", "build"]


def __getattr__(name):
    if name in ("moe", "inputs", "build"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
