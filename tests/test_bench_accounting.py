"""The benchmark's work accounting against the oracle's (CPU only).

bench.py computes active FLOPs for its tokens/s and TFLOP/s figures with its
own formula; the oracle's active_flops is pinned by counting the multiply-adds
of a sparse evaluation of the layer (test_oracle_pins).  The two must agree
on every synthetic workload."""
import pytest

import bench
from grouped_gemm_router_gb300 import inputs
from oracle import moe_oracle as orc


@pytest.mark.parametrize("name", inputs.WORKLOAD_ORDER)
def test_bench_active_flops_match_oracle(name):
    w = inputs.WORKLOADS[name]
    assert bench.active_flops(w) == orc.active_flops(w.T, w.D, w.F, w.E, w.k, w.shared)


def test_w1w3_launch_flops_include_the_shared_rows():
    w = inputs.WORKLOADS["gptoss_lite"]
    routed = orc.w1w3_flops(w.T, w.D, w.F, w.k)
    assert routed == 309_237_645_312
    assert bench.w1w3_flops_per_launch(w) == routed + 4 * w.T * w.D * w.F
