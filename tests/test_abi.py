"""The C ABI library builds for sm_103a, loads, exports every declared entry
point, and rejects bad arguments on the host before any launch (these calls
need no GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_ffn.h")


@pytest.fixture(scope="module")
def native():
    from grouped_gemm_router_gb300 import build
    build.build()
    from grouped_gemm_router_gb300 import _native
    return _native


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:moe_status|size_t|uint64_t|int|const char\s*\*)\s*(moe_\w+)\s*\(",
                                 text, flags=re.M)))


def test_every_declared_symbol_is_exported(native):
    names = declared_functions()
    assert len(names) >= 12
    lib = ctypes.CDLL(native.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in moe_ffn.h but not exported"
    assert set(names) == set(native._SIGNATURES), "binding signatures and header disagree"


def test_status_strings(native):
    assert native.status_str(0) == "ok"
    assert "invalid" in native.status_str(-1)
    assert native.status_str(-99) == "unknown status"


FAKE = 0x100000  # a 16-byte aligned address that is never dereferenced


def _forward(native, d, ws_bytes=1 << 40, x=FAKE, out=FAKE, shared=(None, None, None), ws=FAKE):
    p = ctypes.c_void_p
    return native.lib.moe_ffn_forward(p(x), p(FAKE), None, p(FAKE), p(FAKE), p(FAKE),
                                      *(p(s) if s else None for s in shared), d, p(out), p(ws),
                                      ws_bytes, None, None)


def test_argument_validation_before_launch(native):
    N = native
    good = N.dims(256, 128, 256, 4, 2)
    assert _forward(N, N.dims(0, 128, 256, 4, 2)) == N.MOE_OK           # T = 0: nothing to do
    assert _forward(N, good, x=0) == N.MOE_ERR_INVALID_ARG                # null input
    assert _forward(N, good, out=FAKE + 4) == N.MOE_ERR_INVALID_ARG       # misaligned
    assert _forward(N, N.dims(256, 128, 256, 4, 5)) == N.MOE_ERR_INVALID_ARG   # k > E
    assert _forward(N, N.dims(256, 100, 256, 4, 2)) == N.MOE_ERR_UNSUPPORTED_SHAPE  # D % 64
    assert _forward(N, N.dims(256, 128, 16384, 4, 2)) == N.MOE_ERR_UNSUPPORTED_SHAPE  # F cap
    assert _forward(N, N.dims(256, 128, 256, 200, 2)) == N.MOE_ERR_UNSUPPORTED_SHAPE  # E cap
    assert _forward(N, N.dims(256, 128, 256, 64, 17)) == N.MOE_ERR_UNSUPPORTED_SHAPE  # k cap
    assert _forward(N, good, shared=(FAKE, None, FAKE)) == N.MOE_ERR_INVALID_ARG   # partial shared
    assert _forward(N, good, ws_bytes=100) == N.MOE_ERR_WORKSPACE
    p = ctypes.c_void_p
    assert N.lib.moe_route(None, p(FAKE), None, good, p(FAKE), p(FAKE), None, p(FAKE), 1 << 20,
                           None) == N.MOE_ERR_INVALID_ARG
    assert N.lib.moe_route(p(FAKE), p(FAKE), None, good, p(FAKE), p(FAKE), None, p(FAKE), 16,
                           None) == N.MOE_ERR_WORKSPACE
    assert N.lib.moe_route_scratch_size(N.dims(10, 768, 64, 64, 4)) == 24 * 8 * 32 * 16
    assert N.lib.moe_permute(p(FAKE), good, p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), None,
                             p(FAKE), 1 << 20, None) == N.MOE_ERR_INVALID_ARG   # x without x_sorted
    assert N.lib.moe_permute(p(FAKE), good, p(FAKE), p(FAKE), p(FAKE), p(FAKE), None, None,
                             p(FAKE), 4, None) == N.MOE_ERR_WORKSPACE
    assert N.lib.moe_grouped_swiglu(p(FAKE), None, p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), good,
                                    p(FAKE), None) == N.MOE_ERR_INVALID_ARG     # shared needs x
    assert N.lib.moe_combine(p(FAKE), None, p(FAKE), p(FAKE), N.dims(4, 96, 64, 4, 2), p(FAKE),
                             None) == N.MOE_ERR_UNSUPPORTED_SHAPE
    assert N.lib.moe_grouped_down(p(FAKE), p(FAKE), p(FAKE), p(FAKE), good, p(FAKE), None,
                                  None) == N.MOE_ERR_INVALID_ARG     # the shared expert needs ys
    # the chained kernel keeps a D-column fp32 accumulator in TMEM: D <= 256
    chained = lambda d, x=FAKE, shared=(None, None, None), ys=FAKE: N.lib.moe_grouped_ffn_chained(
        p(FAKE), p(x) if x else None, p(FAKE), p(FAKE), p(FAKE), *(p(s) if s else None for s in shared),
        p(FAKE), d, p(FAKE), p(ys) if ys else None, None)
    assert chained(N.dims(256, 320, 256, 4, 2)) == N.MOE_ERR_UNSUPPORTED_SHAPE
    assert chained(good, x=0, shared=(FAKE, FAKE, FAKE)) == N.MOE_ERR_INVALID_ARG   # shared needs x
    assert chained(good, shared=(FAKE, FAKE, None)) == N.MOE_ERR_INVALID_ARG        # partial shared
    assert chained(good, shared=(FAKE, FAKE, FAKE), ys=0) == N.MOE_ERR_INVALID_ARG  # shared needs ys
    assert chained(N.dims(0, 128, 256, 4, 2)) == N.MOE_OK
    opts = N.MoeOptions()
    opts.flags = N.MOE_FFN_CHAINED
    fwd = lambda d, o: N.lib.moe_ffn_forward(p(FAKE), p(FAKE), None, p(FAKE), p(FAKE), p(FAKE), None,
                                             None, None, d, p(FAKE), p(FAKE), 1 << 40, ctypes.byref(o),
                                             None)
    assert fwd(N.dims(256, 512, 256, 4, 2), opts) == N.MOE_ERR_UNSUPPORTED_SHAPE
    opts.flags = 2   # no such flag
    assert fwd(good, opts) == N.MOE_ERR_INVALID_ARG
    assert N.lib.moe_selftest_wait_timeout(0, p(FAKE), None) == N.MOE_ERR_INVALID_ARG
    assert N.lib.moe_selftest_wait_timeout(10, None, None) == N.MOE_ERR_INVALID_ARG
    assert N.lib.moe_launch_count() == 0


def test_backward_argument_validation_before_launch(native):
    N = native
    p = ctypes.c_void_p
    good = N.dims(256, 128, 256, 4, 2)
    fws = N.lib.moe_ffn_workspace_size(good, 0, 0)
    bws = N.lib.moe_ffn_backward_workspace_size(good, 0)

    def bwd_call(d=good, d_out=FAKE, fwd_bytes=fws, ws_bytes=bws, shared=(None, None, None),
                 dshared=(None, None, None), opts=None):
        ptr = lambda v: p(v) if v else None
        return N.lib.moe_ffn_backward(p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), *map(ptr, shared),
                                      ptr(d_out), d, p(FAKE), fwd_bytes, p(FAKE), None, None, p(FAKE), p(FAKE),
                                      p(FAKE), *map(ptr, dshared), p(FAKE), ws_bytes,
                                      ctypes.byref(opts) if opts else None, None)

    assert bwd_call(d=N.dims(0, 128, 256, 4, 2)) == N.MOE_OK              # nothing to do
    assert bwd_call(d_out=0) == N.MOE_ERR_INVALID_ARG                     # no incoming gradient
    assert bwd_call(shared=(FAKE, FAKE, FAKE)) == N.MOE_ERR_INVALID_ARG   # shared weights, no gradients
    assert bwd_call(dshared=(FAKE, FAKE, FAKE)) == N.MOE_ERR_INVALID_ARG  # gradients, no shared weights
    assert bwd_call(fwd_bytes=fws - 1) == N.MOE_ERR_WORKSPACE
    assert bwd_call(ws_bytes=bws - 1) == N.MOE_ERR_WORKSPACE
    assert bwd_call(d=N.dims(256, 100, 256, 4, 2)) == N.MOE_ERR_UNSUPPORTED_SHAPE
    o = N.MoeOptions()
    o.flags = 2
    assert bwd_call(opts=o) == N.MOE_ERR_INVALID_ARG                      # no such flag
    assert N.lib.moe_launch_count() == 0


def test_backward_workspace_size_matches_documented_layout(native):
    a = lambda n: (n + 255) // 256 * 256
    for T, D, F, E, k, sh in [(256, 128, 256, 4, 2, 0), (32768, 768, 1536, 8, 2, 1), (1, 64, 64, 1, 1, 1)]:
        S = T * k
        Sp = S + 64 * E
        R = Sp + (T if sh else 0)
        n = a(Sp * D * 2) + a(R * F * 2) + a(R * F * 4) + a(R * F * 2) + a(R * D * 2) + 2 * a(S * 4)
        n += a((S // 64 + E) * (D + 1) * 4) + a(E * D * 2)
        kb = (S + 64 * E) // 64 + ((T + 63) // 64 if sh else 0)     # weight-gradient partial slots
        n += a((kb // 80 + 2) * 2 * D * F * 4)
        assert native.lib.moe_ffn_backward_workspace_size(native.dims(T, D, F, E, k), sh) == n


def test_workspace_size_matches_documented_layout(native):
    def layout(T, D, F, E, k, shared, host_io):
        a = lambda n: (n + 255) // 256 * 256
        S = T * k
        rows = S + (T if shared else 0)
        nblk = (T + 15) // 16        # histogram rows for the smallest block (16 tokens)
        et = (E + 7) // 8
        et = et if et <= 2 else 4 if et <= 4 else 8 if et <= 8 else 16
        n = a((D // 32) * et * 32 * 16) + a(S * 4) * 2 + a(nblk * E * 4) + a(E * 4) + a((E + 1) * 4) + a(S * 4) * 2
        n += a(S * D * 2) + a(rows * F * 2) + a(S * D * 2) + (a(T * D * 4) if shared else 0)
        if host_io:
            n += 2 * a(T * D * 2)
        return n

    for T, D, F, E, k, sh, hio in [(256, 128, 256, 4, 2, 0, 0), (32768, 768, 1536, 8, 2, 1, 1),
                                   (2048, 768, 1536, 64, 4, 1, 0), (1, 64, 64, 1, 1, 0, 1)]:
        assert native.lib.moe_ffn_workspace_size(native.dims(T, D, F, E, k), sh, hio) == \
            layout(T, D, F, E, k, sh, hio)
    assert native.lib.moe_ffn_workspace_size(native.dims(10, 100, 64, 4, 2), 0, 0) == 0


def test_permute_scratch_covers_every_device(native):
    # sized for 16-token blocks, the most histogram rows any device uses
    for T, E in [(1, 4), (2048, 64), (32768, 8), (65536, 128)]:
        assert native.lib.moe_permute_scratch_size(native.dims(T, 64, 64, E, 1)) == (T + 15) // 16 * E * 4


def test_product_path_fails_loudly_without_library(tmp_path):
    from grouped_gemm_router_gb300 import _native
    with pytest.raises(ImportError):
        _native.load(str(tmp_path / "missing.so"))
