"""The allocation-free permutation entry point, moe_permute_noalloc.

It serves callers that cannot allocate device memory: its block-histogram
scratch is a fixed array inside the library instead of a caller buffer.  This
test calls it through the C ABI twice in a row (the second call runs on the
array the first call left behind) and checks that its results equal those of
moe_permute, the entry point that takes a caller-provided scratch buffer.
Counts, offsets, the permutation, its inverse and the gathered rows are
integer / byte results, so the comparison is exact.  The file name makes
pytest collect it last."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def native():
    from grouped_gemm_router_gb300 import build
    build.build()
    from grouped_gemm_router_gb300 import _native
    return _native


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _permute_with_scratch(N, ids, E, x):
    T, k = ids.shape
    D = x.shape[1]
    d = N.dims(T, D, 64, E, k)
    S = T * k
    out = {n: torch.empty(E if n == "counts" else E + 1 if n == "offsets" else S,
                          dtype=torch.int32, device="cuda") for n in ("counts", "offsets", "perm", "inv")}
    out["x_sorted"] = torch.empty(S, D, dtype=torch.bfloat16, device="cuda")
    nscr = int(N.lib.moe_permute_scratch_size(d))
    scratch = torch.empty(nscr, dtype=torch.uint8, device="cuda")
    st = N.lib.moe_permute(_p(ids), d, _p(out["counts"]), _p(out["offsets"]), _p(out["perm"]),
                           _p(out["inv"]), _p(x), _p(out["x_sorted"]), _p(scratch), nscr, None)
    N.check(st, "moe_permute")
    return out


def _permute_noalloc(N, ids, E, x):
    T, k = ids.shape
    D = x.shape[1]
    S = T * k
    # poison the outputs so that stale values cannot pass
    out = {n: torch.full((E if n == "counts" else E + 1 if n == "offsets" else S,), -7,
                         dtype=torch.int32, device="cuda") for n in ("counts", "offsets", "perm", "inv")}
    out["x_sorted"] = torch.zeros(S, D, dtype=torch.bfloat16, device="cuda")
    st = N.lib.moe_permute_noalloc(_p(ids), N.dims(T, D, 64, E, k), _p(out["counts"]), _p(out["offsets"]),
                                   _p(out["perm"]), _p(out["inv"]), _p(x), _p(out["x_sorted"]), None)
    N.check(st, "moe_permute_noalloc")
    return out


def _case(T, E, k, seed):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    x = rng.integers(-2 ** 15, 2 ** 15, size=(T, 128), dtype=np.int64).astype(np.int16)
    return torch.from_numpy(ids).cuda(), torch.from_numpy(x).view(torch.bfloat16).cuda()


def test_noalloc_matches_scratch_entry_on_two_calls_in_a_row(native):
    N = native
    # two different problems back to back: the second call sees the first
    # call's histogram still in the shared array
    for T, E, k, seed in [(32768, 8, 2, 1), (2000, 64, 4, 2)]:
        ids, x = _case(T, E, k, seed)
        ref = _permute_with_scratch(N, ids, E, x)
        got = _permute_noalloc(N, ids, E, x)
        torch.cuda.synchronize()
        for name in ("counts", "offsets", "perm", "inv"):
            assert torch.equal(got[name], ref[name]), f"{name} differs (T={T}, E={E})"
        assert torch.equal(got["x_sorted"].view(torch.int16), ref["x_sorted"].view(torch.int16))


def test_noalloc_at_the_size_limit(native):
    """With 16-token histogram blocks, T = 8192 and E = 128 need exactly the
    65,536 entries the array holds: accepted, and equal to moe_permute.  Sixteen
    more tokens need one more block row: rejected before anything runs."""
    N = native
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if 32 * 2 * sms <= 8208:
        pytest.skip("16-token blocks need more SMs than this device has at T = 8208")
    E, k = 128, 1
    need = lambda T: -(-T // int(N.lib.moe_route_block_tokens(T))) * E
    assert need(8192) == 65536 and need(8208) == 65536 + E
    ids, x = _case(8192, E, k, 3)
    ref = _permute_with_scratch(N, ids, E, x)
    got = _permute_noalloc(N, ids, E, x)
    torch.cuda.synchronize()
    for name in ("counts", "offsets", "perm", "inv"):
        assert torch.equal(got[name], ref[name]), name
    assert torch.equal(got["x_sorted"].view(torch.int16), ref["x_sorted"].view(torch.int16))
    fake = ctypes.c_void_p(0x100000)
    st = N.lib.moe_permute_noalloc(fake, N.dims(8208, 128, 64, E, k), fake, fake, fake, fake, None, None, None)
    assert st == N.MOE_ERR_UNSUPPORTED_SHAPE


def test_noalloc_rejects_sizes_beyond_its_array(native):
    N = native
    T, E, k = 65 * 1024, 128, 1          # 64-token blocks: ceil(T/64) * E = 133,120 > 65,536
    fake = ctypes.c_void_p(0x100000)
    st = N.lib.moe_permute_noalloc(fake, N.dims(T, 64, 64, E, k), fake, fake, fake, fake, None, None, None)
    assert st == N.MOE_ERR_UNSUPPORTED_SHAPE
