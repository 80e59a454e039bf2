"""Multi-rank host logic on CPU with the gloo backend (world size 2).

The layer partitions by tokens: with the weights replicated, each token's
output depends only on its own row, so ranks can run independent replicas on
their own batches with no collective on the data path.  These tests check
that property on the oracle (sharded == unsharded), the max-over-ranks step
time that bench.py reports, and that the reference arm prints one line from
rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from grouped_gemm_router_gb300 import inputs
    from oracle import moe_oracle as orc

    # 1. token-sharded oracle: each rank runs its half of the tokens
    w = inputs.WORKLOADS["tiny"]
    L = inputs.make_layer(w)
    T = w.T
    lo, hi = rank * T // world, (rank + 1) * T // world
    out = orc.moe_ffn_forward(L["x"][lo:hi], L["Wg"], L["W1"], L["W3"], L["W2"], w.k, bias=L["bias"])
    parts = [None] * world
    dist.all_gather_object(parts, out)
    # 2. the benchmark's step time is the max over ranks
    m = bench.reduce_max(1.5 + rank, "cpu")
    if rank == 0:
        np.save(os.path.join(out_dir, "sharded.npy"), np.concatenate(parts))
        with open(os.path.join(out_dir, "max.json"), "w") as f:
            json.dump({"max": m}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_token_sharded_replicas_match_unsharded_and_max_over_ranks(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    sys.path.insert(0, ROOT)
    from grouped_gemm_router_gb300 import inputs
    from oracle import moe_oracle as orc
    w = inputs.WORKLOADS["tiny"]
    L = inputs.make_layer(w)
    full = orc.moe_ffn_forward(L["x"], L["Wg"], L["W1"], L["W3"], L["W2"], w.k, bias=L["bias"])
    sharded = np.load(tmp_path / "sharded.npy")
    assert sharded.shape == full.shape
    assert np.abs(sharded - full).max() <= 1e-12 * np.abs(full).max()
    assert json.load(open(tmp_path / "max.json"))["max"] == 2.5


def test_reference_arm_prints_one_line_from_rank0():
    env = dict(os.environ, PYTHONPATH=ROOT)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "1", "--workload", "tiny"]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
