"""Benchmark of the MoE SwiGLU FFN forward pass on GB300.

A step is one forward pass of the whole layer (router -> top-k/softmax ->
stable permutation -> W1||W3 + SiLU*mul -> W2 -> weighted combine, plus the
shared expert) over one batch of synthetic tokens of the GPT-OSS-Lite-shaped
workload (T=32768, D=768, F=1536, E=8 routed top-2 + 1 shared expert), with
all inputs resident in HBM.  One JSON line is printed by rank 0.  On one GPU
the line also carries `per_workload`: the same measurement (tokens/s, active
TFLOP/s, roofline placement, stage times, clocks) for each of the other
synthetic workloads (tiny, skewed, small_chunk, wide), with the same steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

Timing: W untimed warm-up steps; then K steps, each bracketed by CUDA events
on the launching stream.  Between steps (outside the events) a 512 MB buffer
is written and then read back, so each step starts with a cold L2 that holds
no dirty lines of the flush (their write-back is not charged to the step).
Multi-GPU (torchrun): every rank runs its own replica of the layer on its own
batch (weak scaling, no collective on the data path); the step time is the max
over ranks.

--impl reference times the fp64 CPU oracle as it stands on the host cores
(rank 0 only), every step on the first n tokens of the same workload with n
sized so the run takes about a minute and a half, and prints the same line
with "impl": "reference" and the time of the steps it actually ran.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from grouped_gemm_router_gb300 import inputs  # noqa: E402

WORKLOAD = "gptoss_lite"
DATASHEET_BF16_DENSE_TFLOPS = 2250.0  # GB300 dense bf16 (the datasheet's sparse figure halved)
METRIC = "MoE FFN fwd tokens/s and active TFLOP/s on 1 GB300; % of bf16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
REF_BUDGET_S = 90.0  # wall time of the reference arm's warm-up + timed steps


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def active_flops(w) -> int:
    """Router GEMM + routed W1/W3/W2 + shared-expert W1/W3/W2 (2 FLOPs per MAC)."""
    return (2 * w.T * w.D * w.E + 6 * w.T * w.k * w.D * w.F
            + (6 * w.T * w.D * w.F if w.shared else 0))


def w1w3_flops_per_launch(w) -> int:
    """Algorithmic FLOPs of one launch of the W1||W3 grouped GEMM: each routed
    slot and (with the shared expert) each token does two [D]x[D,F] products."""
    rows = w.T * w.k + (w.T if w.shared else 0)
    return 4 * rows * w.D * w.F


def stage_bytes(w) -> dict:
    """Algorithmic HBM bytes per stage (each tensor read or written once)."""
    T, D, F, E, k = w.T, w.D, w.F, w.E, w.k
    S = T * k
    rows = S + (T if w.shared else 0)
    sh = 1 if w.shared else 0
    return {
        "route": T * D * 2 + D * E * 2 + S * 8,
        "permute": T * D * 2 + S * D * 2 + S * 4 * 3,
        "w1w3": S * D * 2 + sh * T * D * 2 + (E + sh) * 2 * D * F * 2 + rows * F * 2,
        # the shared expert's rows of the down-projection (ys) are fp32
        "w2": rows * F * 2 + (E + sh) * F * D * 2 + S * D * 2 + sh * T * D * 4,
        "combine": S * D * 2 + sh * T * D * 4 + T * D * 2 + S * 8,
    }


def source_hash() -> str:
    """Hash of the sources of the dominant kernel (the forward grouped GEMM and
    the device helpers it includes): the committed ncu traffic is valid only
    for the kernel built from these exact files."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "grouped_gemm_router_gb300", "csrc")
    for n in ("grouped_gemm.cu", "moe_device.cuh"):
        h.update(open(os.path.join(csrc, n), "rb").read())
    return h.hexdigest()[:16]


def w1w3_kernel_name(w):
    """The W1||W3 kernel instance the library launches for this layer: it
    stages 128 k per stage when D is a multiple of 128, 64 k otherwise."""
    return "grouped_gemm_pair_kernel<true, true>" if w.D % 128 == 0 else "grouped_gemm_pair_kernel<true, false>"


def ncu_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or
    None when the kernels changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("source_hash") != source_hash():
        return None
    v = d.get("kernels", {}).get(kernel)
    return None if v is None else float(v)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *a):
        pass

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def reduce_max(value: float, device) -> float:
    """Max of a per-rank value over all ranks (the value itself without a
    process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def to_dev(a, dev):
    import torch
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(a).to(dev)


def time_oracle(L, w, budget_s=12.0):
    """Times the fp64 oracle on the first n tokens of the workload, growing n
    until one run takes about a second, then repeats within the budget.
    Returns (tokens/s, n tokens per run, runs, seconds)."""
    from oracle import moe_oracle as orc
    n = 64
    while True:
        t0 = time.perf_counter()
        orc.moe_ffn_forward(L["x"][:n], L["Wg"], L["W1"], L["W3"], L["W2"], w.k, bias=L["bias"],
                            Ws1=L["Ws1"], Ws3=L["Ws3"], Ws2=L["Ws2"])
        dt = time.perf_counter() - t0
        if dt > 1.0 or n >= w.T:
            break
        n = min(w.T, n * 4)
    runs, total, t_start = 0, 0.0, time.perf_counter()
    while time.perf_counter() - t_start < budget_s - dt or runs == 0:
        t0 = time.perf_counter()
        orc.moe_ffn_forward(L["x"][:n], L["Wg"], L["W1"], L["W3"], L["W2"], w.k, bias=L["bias"],
                            Ws1=L["Ws1"], Ws3=L["Ws3"], Ws2=L["Ws2"])
        total += time.perf_counter() - t0
        runs += 1
    return n * runs / total, n, runs, total


def near_tie_tokens(L, w) -> int:
    """Tokens whose k-th and (k+1)-th fp64 oracle logits differ by less than
    1e-3: there either selection is correct (the parity tests' near-tie rule)."""
    from oracle import moe_oracle as orc
    logits = orc.router_logits(orc.bf16_to_f64(L["x"]), orc.bf16_to_f64(L["Wg"]), L["bias"])
    return int((orc.topk_gap(logits, w.k) < 1e-3).sum())


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


L2_NOTE = "flushed between steps (512 MB write + read back)"


def line_config(w, world: int) -> dict:
    """The `config` object of both arms' JSON lines (identical for the same run)."""
    return {"workload": w.name, "T": w.T, "D": w.D, "F": w.F, "E": w.E, "k": w.k,
            "shared_expert": w.shared, "l2": L2_NOTE, "parallelism": f"replicas x{world}"}


def run_reference(args, w, rank, world):
    """The reference arm: the fp64 oracle as it stands, on the host cores.
    Every step runs the whole layer on the first n tokens of the workload; n
    is sized from a calibration run so that the warm-up and timed steps take
    about REF_BUDGET_S together (n = T when that fits).  The line reports the
    time of the steps actually run: ms_per_step is one n-token step, value is
    n tokens / that time."""
    if rank != 0:
        return
    from oracle import moe_oracle as orc
    L = inputs.make_layer(w)

    def run(n):
        orc.moe_ffn_forward(L["x"][:n], L["Wg"], L["W1"], L["W3"], L["W2"], w.k, bias=L["bias"],
                            Ws1=L["Ws1"], Ws3=L["Ws3"], Ws2=L["Ws2"])

    # calibration: a step costs about fixed + per_token * n seconds
    cal = []
    for n_cal in (min(w.T, 256), min(w.T, 1024)):
        t0 = time.perf_counter()
        run(n_cal)
        cal.append((n_cal, time.perf_counter() - t0))
    (n1, t1), (n2, t2) = cal
    per_token = (t2 - t1) / (n2 - n1) if n2 > n1 else t2 / n2
    per_token = max(per_token, t2 / n2 / 4)
    fixed = max(0.0, t2 - per_token * n2)
    nsteps = max(1, args.steps) + max(0, args.warmup)
    n = int((REF_BUDGET_S / nsteps - fixed) / per_token) // 64 * 64
    n = max(min(64, w.T), min(w.T, n))
    for _ in range(args.warmup):
        run(n)
    times = []
    for _ in range(max(1, args.steps)):
        t0 = time.perf_counter()
        run(n)
        times.append(time.perf_counter() - t0)
    step_s = float(np.mean(times))
    tps = n / step_s
    sample = (f"the first {n} of the workload's {w.T} tokens through the whole layer per step "
              f"(fp64 numpy oracle); {len(times)} timed steps")
    line = {
        "impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": len(times), "warmup": args.warmup, "ms_per_step": 1e3 * step_s,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": line_config(w, world), "sample_tokens": n,
        "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": host_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_sweep(args):
    """Roofline placement of the two grouped GEMMs as F/D and the tokens per
    expert vary (the sweeps the Chinchilla/MoE page recommends for placing
    the MoE FFN on the roofline).  One JSON line per shape."""
    import torch
    from grouped_gemm_router_gb300 import build
    build.build()
    from grouped_gemm_router_gb300 import moe

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pk, pk_kind = peaks()
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    E, k = 8, 2
    shapes = []
    if args.sweep in ("fd", "all"):   # F/D at a fixed 8192 tokens per expert
        shapes += [("fd", 32768, 768, F) for F in (384, 768, 1536, 3072, 6144)]
    if args.sweep in ("t", "all"):    # tokens per expert t = T*k/E at D=768, F=1536
        shapes += [("t", T, 768, 1536) for T in (256, 1024, 4096, 16384, 65536)]
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    for kind, T, D, F in shapes:
        w, L = inputs.make_custom(T, D, F, E, k, False, 7)
        G = {key: to_dev(v, dev) for key, v in L.items()}
        ws = moe.Workspace(T, D, F, E, k, False, device=dev)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
        for row in evs:
            for ev in row:
                ev.record()
        for _ in range(args.warmup):
            moe.moe_ffn_forward(G["x"], G["Wg"], G["W1"], G["W3"], G["W2"], k, workspace=ws)
        for i in range(args.steps):
            flush.fill_(1.0)
            moe.moe_ffn_forward(G["x"], G["Wg"], G["W1"], G["W3"], G["W2"], k, workspace=ws,
                                stage_events=evs[i])
        torch.cuda.synchronize()
        t13 = float(np.mean([evs[i][2].elapsed_time(evs[i][3]) for i in range(args.steps)])) / 1e3
        t2 = float(np.mean([evs[i][3].elapsed_time(evs[i][4]) for i in range(args.steps)])) / 1e3
        S = T * k
        t = S / E
        # algorithmic work: each tensor read or written once
        fl13, fl2 = 4 * S * D * F, 2 * S * F * D
        by13 = S * D * 2 + 2 * E * D * F * 2 + S * F * 2
        by2 = S * F * 2 + E * F * D * 2 + S * D * 2
        line = {"sweep": kind, "T": T, "D": D, "F": F, "E": E, "k": k, "tokens_per_expert": t,
                "F_over_D": F / D,
                "w1w3": {"us": t13 * 1e6, "tflops": fl13 / t13 / 1e12, "gbs": by13 / t13 / 1e9,
                         "intensity": fl13 / by13, "frac_tensor": fl13 / t13 / 1e12 / pk["bf16_tflops"],
                         "frac_hbm": by13 / t13 / 1e9 / pk["hbm_gbs"]},
                "w2": {"us": t2 * 1e6, "tflops": fl2 / t2 / 1e12, "gbs": by2 / t2 / 1e9,
                       "intensity": fl2 / by2, "frac_tensor": fl2 / t2 / 1e12 / pk["bf16_tflops"],
                       "frac_hbm": by2 / t2 / 1e9 / pk["hbm_gbs"]},
                # the page's per-expert traffic model of the unfused up / down pair
                "page_unfused_bytes_per_expert": 4 * t * D + 4 * t * F + 4 * D * F,
                "page_fused_bytes_per_expert": 4 * t * D + 4 * D * F,
                "ridge_flop_per_byte": ridge, "peaks": pk_kind}
        print(json.dumps(line), flush=True)
        del G, ws


def run_chain_sweep(args):
    """Chained (h kept on chip) vs unchained (h through HBM) expert FFN as F/D
    and the tokens per expert vary: the sweeps the fused-Triton-kernel page
    proposes to place the fused kernel on the roofline.  One JSON line per
    shape; times are CUDA events around the expert stage(s) of the layer."""
    import torch
    from grouped_gemm_router_gb300 import build
    build.build()
    from grouped_gemm_router_gb300 import moe

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pk, pk_kind = peaks()
    E, k = 8, 2
    shapes = [("chain_fd", 2048, 256, F) for F in (256, 512, 1024, 2048, 4096)]
    shapes += [("chain_fd", 32768, 256, F) for F in (256, 1024, 4096)]
    shapes += [("chain_t", T, 256, 1024) for T in (256, 1024, 4096, 16384, 65536)]
    shapes += [("chain_t", T, 128, 1024) for T in (1024, 16384)]
    if args.chain_shape:  # one shape, e.g. for a DRAM-counter capture
        T, D, F = (int(v) for v in args.chain_shape.split("x"))
        shapes = [("chain_one", T, D, F)]
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)
    for kind, T, D, F in shapes:
        w, L = inputs.make_custom(T, D, F, E, k, False, 7)
        G = {key: to_dev(v, dev) for key, v in L.items()}
        ws = moe.Workspace(T, D, F, E, k, False, device=dev)
        res = {}
        for chained in (False, True):
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
            for row in evs:
                for ev in row:
                    ev.record()
            for _ in range(args.warmup):
                moe.moe_ffn_forward(G["x"], G["Wg"], G["W1"], G["W3"], G["W2"], k, workspace=ws,
                                    chained=chained)
            for i in range(args.steps):
                flush.fill_(1.0)
                sink.copy_(flush.sum())
                moe.moe_ffn_forward(G["x"], G["Wg"], G["W1"], G["W3"], G["W2"], k, workspace=ws,
                                    stage_events=evs[i], chained=chained)
            torch.cuda.synchronize()
            res[chained] = float(np.mean([evs[i][2].elapsed_time(evs[i][4]) for i in range(args.steps)])) / 1e3
        assert moe.device_error() == 0
        S = T * k
        t = S / E
        flops = 6 * S * D * F
        fused_bytes = S * D * 2 + 3 * E * D * F * 2 + S * D * 2
        unfused_bytes = fused_bytes + 2 * S * F * 2
        line = {"sweep": kind, "T": T, "D": D, "F": F, "E": E, "k": k, "tokens_per_expert": t,
                "F_over_D": F / D,
                "unchained_us": res[False] * 1e6, "chained_us": res[True] * 1e6,
                "speedup": res[False] / res[True],
                "unchained_tflops": flops / res[False] / 1e12, "chained_tflops": flops / res[True] / 1e12,
                "unchained_frac_tensor": flops / res[False] / 1e12 / pk["bf16_tflops"],
                "chained_frac_tensor": flops / res[True] / 1e12 / pk["bf16_tflops"],
                "intensity_unfused": flops / unfused_bytes, "intensity_fused": flops / fused_bytes,
                "unfused_bytes": unfused_bytes, "fused_bytes": fused_bytes,
                # the page's model of the speedup while memory-bound
                "page_model_speedup": 1 + t * F / (t * D + D * F),
                "ridge_flop_per_byte": pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9), "peaks": pk_kind}
        print(json.dumps(line), flush=True)
        del G, ws


def run_backward_bench(args, w):
    """Training step of the layer: forward then backward (d_out synthetic),
    L2 flushed before each step.  One JSON line: tokens/s of forward +
    backward, the backward's stage times and each backward GEMM's rate."""
    import torch
    from grouped_gemm_router_gb300 import build
    build.build()
    from grouped_gemm_router_gb300 import moe

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pk, pk_kind = peaks()
    L = inputs.make_layer(w)
    G = {key: to_dev(v, dev) for key, v in L.items()}
    T, D, F, E, k = w.T, w.D, w.F, w.E, w.k
    rng = np.random.default_rng(1)
    d_out = to_dev(inputs.f32_to_bf16_bits(rng.standard_normal((T, D)).astype(np.float32)), dev)
    ws = moe.Workspace(T, D, F, E, k, w.shared, device=dev)
    bws = moe.BackwardWorkspace(T, D, F, E, k, w.shared, device=dev)
    out = torch.empty(T, D, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)
    sh = dict(Ws1=G["Ws1"], Ws3=G["Ws3"], Ws2=G["Ws2"]) if w.shared else {}

    def step(fev=None, bev=None):
        moe.moe_ffn_forward(G["x"], G["Wg"], G["W1"], G["W3"], G["W2"], k, bias=G["bias"], out=out,
                            workspace=ws, stage_events=fev, **sh)
        return moe.moe_ffn_backward(G["x"], G["Wg"], G["W1"], G["W3"], G["W2"], k, d_out, ws,
                                    bwd_workspace=bws, stage_events=bev, **sh)

    nb = max(args.steps, 1)
    fevs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(nb)]
    bevs = [[torch.cuda.Event(enable_timing=True) for _ in range(9)] for _ in range(nb)]
    for row in fevs + bevs:
        for ev in row:
            ev.record()
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    with ClockSampler(0) as cs:
        for i in range(nb):
            flush.fill_(1.0)
            sink.copy_(flush.sum())
            step(fevs[i], bevs[i])
        torch.cuda.synchronize()
        clocks = cs.stop()
    assert moe.device_error() == 0
    mean = lambda evs, a, b: float(np.mean([e[a].elapsed_time(e[b]) for e in evs])) / 1e3
    fwd_s = mean(fevs, 0, 5)
    bwd_s = mean(bevs, 0, 8)
    R = T * k + (T if w.shared else 0)
    names = ["combine_bwd", "w2_dgrad", "swiglu_bwd_recompute", "x_dgrad", "wgrad_w1w3", "wgrad_w2",
             "dx_gather", "router_bwd"]
    stage = {n: mean(bevs, i, i + 1) * 1e3 for i, n in enumerate(names)}
    flops = {"w2_dgrad": 2 * R * D * F, "swiglu_bwd_recompute": 4 * R * D * F, "x_dgrad": 4 * R * D * F,
             "wgrad_w1w3": 4 * R * D * F, "wgrad_w2": 2 * R * D * F}
    bwd_flops = sum(flops.values()) + 2 * T * D * E
    line = {"metric": "MoE FFN forward + backward tokens/s on 1 GB300", "value": T / (fwd_s + bwd_s),
            "unit": "tokens/s", "steps": nb, "warmup": max(args.warmup, 3), "dtype": "bf16",
            "data": "synthetic", "config": {"workload": w.name, "T": T, "D": D, "F": F, "E": E, "k": k,
                                            "shared_expert": w.shared,
                                            "l2": "flushed before each step (512 MB write + read back)"},
            "fwd_ms": fwd_s * 1e3, "bwd_ms": bwd_s * 1e3,
            "fwd_tflops": active_flops(w) / fwd_s / 1e12, "bwd_tflops": bwd_flops / bwd_s / 1e12,
            "bwd_stage_ms": stage,
            "bwd_gemm_frac_of_bf16_peak": {n: f / (stage[n] / 1e3) / 1e12 / pk["bf16_tflops"]
                                           for n, f in flops.items()},
            "peak": {"bf16_tflops": pk["bf16_tflops"], "kind": pk_kind}, "clocks": clocks,
            "bwd_launches_per_step": 9}
    print(json.dumps(line), flush=True)


def time_forward(step, flush_l2, K, W, local_rank, world, dev, moe):
    """W warm-up steps, then K timed steps (L2 flushed before each, outside
    the events), then extra steps with an event at every stage boundary for
    the per-stage breakdown.  The timed steps record only a start and an end
    event: events between the kernels would re-serialise their programmatic
    (overlapped) launches.  Returns the mean step time (max over ranks), the
    per-step times, the mean stage times and the clocks seen."""
    import torch
    import torch.distributed as dist
    for _ in range(W):
        flush_l2()
        step()
    torch.cuda.synchronize()
    if moe.device_error() != 0:
        raise RuntimeError("device wait timed out during warm-up")
    step_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    KB = max(3, min(K, 50))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(KB)]
    for row in step_ev + evs:  # create the CUDA events now, outside the timed loop
        for ev in row:
            ev.record()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank).__enter__()
    n_launch0 = moe.launch_count()
    wall0 = time.perf_counter()
    for i in range(K):
        flush_l2()
        step([step_ev[i][0], None, None, None, None, step_ev[i][1]])
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    n_launch = moe.launch_count() - n_launch0
    clocks = sampler.stop()
    if world > 1:
        dist.barrier()
    if moe.device_error() != 0:
        raise RuntimeError("device wait timed out during the timed steps")
    step_ms = np.array([step_ev[i][0].elapsed_time(step_ev[i][1]) for i in range(K)])
    ms = reduce_max(float(step_ms.mean()), dev)
    for i in range(KB):
        flush_l2()
        step(evs[i])
    torch.cuda.synchronize()
    st = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(5)] for i in range(KB)])
    names = ["route", "permute", "w1w3", "w2", "combine"]
    return {"ms": ms, "step_ms": step_ms, "stage_ms": {n: float(st[:, j].mean()) for j, n in enumerate(names)},
            "clocks": clocks, "launches": n_launch, "wall_s": wall, "stage_steps": KB}


def roofline_place(w, ms: float, pk: dict) -> dict:
    """Where one forward step of workload w sits against its roofline: the
    slower of the active FLOPs at the bf16 peak and the algorithmic bytes
    (unchained path, every tensor read or written once) at the HBM peak."""
    fl = active_flops(w)
    by = sum(stage_bytes(w).values())
    t_flop = fl / (pk["bf16_tflops"] * 1e12)
    t_hbm = by / (pk["hbm_gbs"] * 1e9)
    s = ms / 1e3
    return {"bound": "tensor" if t_flop >= t_hbm else "hbm", "roofline_us": 1e6 * max(t_flop, t_hbm),
            "frac": max(t_flop, t_hbm) / s, "frac_tensor": t_flop / s, "frac_hbm": t_hbm / s,
            "active_gflop": fl / 1e9, "algorithmic_mb": by / 1e6}


def measure_other_workloads(names, args, dev, moe, flush_l2, pk) -> dict:
    """Forward-pass tokens/s, active TFLOP/s and roofline placement of each
    named workload (1 GPU), timed like the headline workload."""
    import torch
    res = {}
    for name in names:
        w = inputs.WORKLOADS[name]
        t_gen = time.perf_counter()
        L = inputs.make_layer(w)
        G = {key: to_dev(v, dev) for key, v in L.items()}
        del L
        t_gen = time.perf_counter() - t_gen
        ws = moe.Workspace(w.T, w.D, w.F, w.E, w.k, w.shared, device=dev)
        out = torch.empty(w.T, w.D, dtype=torch.bfloat16, device=dev)

        def step(events=None, G=G, ws=ws, out=out, w=w):
            moe.moe_ffn_forward(G["x"], G["Wg"], G["W1"], G["W3"], G["W2"], w.k, bias=G["bias"],
                                Ws1=G["Ws1"], Ws3=G["Ws3"], Ws2=G["Ws2"], out=out, workspace=ws,
                                stage_events=events)

        tm = time_forward(step, flush_l2, args.steps, args.warmup, 0, 1, dev, moe)
        ms = tm["ms"]
        res[name] = {
            "T": w.T, "D": w.D, "F": w.F, "E": w.E, "k": w.k, "shared_expert": w.shared,
            "value": w.T / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
            "ms_per_step_median": float(np.median(tm["step_ms"])), "steps": args.steps,
            "active_tflops": active_flops(w) / (ms / 1e3) / 1e12,
            "roofline": roofline_place(w, ms, pk), "stage_ms": tm["stage_ms"], "clocks": tm["clocks"],
            "gpu_launches": int(tm["launches"]), "input_generation_s": t_gen,
        }
        del G, ws, out, step
        torch.cuda.empty_cache()
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=list(inputs.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-streams", type=int, default=4,
                    help="streams (each with its own workspace) in the end-to-end host-buffer loop")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip timing the other synthetic workloads after the headline one")
    ap.add_argument("--sweep", choices=["fd", "t", "all", "chained"], default=None,
                    help="roofline placement of the grouped GEMMs over F/D or tokens per expert; "
                         "'chained': chained vs unchained expert FFN (D <= 256)")
    ap.add_argument("--chain-shape", default=None, metavar="TxDxF",
                    help="with --sweep chained: measure this one shape only")
    ap.add_argument("--backward", action="store_true",
                    help="time the training step (forward + backward) instead of the forward")
    args = ap.parse_args()
    if args.backward:
        run_backward_bench(args, inputs.WORKLOADS[args.workload])
        return
    if args.sweep == "chained":
        run_chain_sweep(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.warmup < 3 and args.impl == "native":
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = inputs.WORKLOADS[args.workload]

    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return

    import torch
    import torch.distributed as dist

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    from grouped_gemm_router_gb300 import build
    build.build()
    from grouped_gemm_router_gb300 import moe

    L = inputs.make_layer(w)
    G = {k: to_dev(v, dev) for k, v in L.items()}
    T, D, F, E, k = w.T, w.D, w.F, w.E, w.k
    ws = moe.Workspace(T, D, F, E, k, w.shared, device=dev)
    out = torch.empty(T, D, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    flush_sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2():
        flush.fill_(1.0)
        flush_sink.copy_(flush.sum())

    def step(events=None):
        moe.moe_ffn_forward(G["x"], G["Wg"], G["W1"], G["W3"], G["W2"], k, bias=G["bias"],
                            Ws1=G["Ws1"], Ws3=G["Ws3"], Ws2=G["Ws2"], out=out, workspace=ws,
                            stage_events=events)

    tm = time_forward(step, flush_l2, args.steps, args.warmup, local_rank, world, dev, moe)
    ms, step_ms, stage_ms, clocks = tm["ms"], tm["step_ms"], tm["stage_ms"], tm["clocks"]
    n_launch, wall, KB = tm["launches"], tm["wall_s"], tm["stage_steps"]
    K = args.steps

    # ---- references for the event-timed HBM stages: a plain library read of
    # the same x (torch's float32 sum over its bytes) and an empty launch,
    # each after the same L2 flush ----
    xf = G["x"].view(torch.float32)
    refs = {"torch_sum_x": lambda: xf.sum(), "empty_launch": lambda: torch.cuda._sleep(0)}
    ref_ms = {}
    for name, op in refs.items():
        fev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(KB)]
        for _ in range(3):
            flush_l2()
            op()
        for i in range(KB):
            flush_l2()
            fev[i][0].record()
            op()
            fev[i][1].record()
        torch.cuda.synchronize()
        ref_ms[name] = float(np.mean([fev[i][0].elapsed_time(fev[i][1]) for i in range(KB)]))

    # ---- the same step replayed from a CUDA graph (the L2 flush stays outside) ----
    gs = torch.cuda.Stream(device=dev)
    gs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(gs):
        step()
    torch.cuda.current_stream().wait_stream(gs)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    gev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for row in gev:
        for ev in row:
            ev.record()
    for _ in range(3):
        flush_l2()
        graph.replay()
    torch.cuda.synchronize()
    for i in range(K):
        flush_l2()
        gev[i][0].record()
        graph.replay()
        gev[i][1].record()
    torch.cuda.synchronize()
    graph_ms = reduce_max(float(np.mean([gev[i][0].elapsed_time(gev[i][1]) for i in range(K)])), dev)
    del graph

    # ---- end to end through the host-memory entry point ----
    # args.e2e_streams streams, each with its own workspace and pinned x / out
    # buffers: while one batch computes, the others' x are copied in and their
    # out copied back, as a serving loop would run it.  A stream's own copies
    # and layer run in order, so with two streams a stream's D2H and next H2D
    # (about 0.5 ms together at ~200 GB/s for gptoss_lite) outlast the other
    # stream's layer; with four the copies hide under the layers (gptoss_lite:
    # 520, 508 and 496 us per step with two, three and four).  Every step copies its whole x
    # from pinned host memory and its whole out back to pinned host memory
    # inside the timed region (no L2 flush between these steps); the region
    # also holds the pipeline's fill (first H2D) and drain (last D2H).
    nstream = args.e2e_streams
    streams = [torch.cuda.Stream(device=dev) for _ in range(nstream)]
    ws_h = [moe.Workspace(T, D, F, E, k, w.shared, host_io=True, device=dev) for _ in range(nstream)]
    x_host = [G["x"].cpu().pin_memory() for _ in range(nstream)]
    out_host = [torch.empty(T, D, dtype=torch.bfloat16).pin_memory() for _ in range(nstream)]
    K2 = max(50, min(K, 200))  # fill and drain spread over at least 50 steps

    def e2e_step(i):
        j = i % nstream
        with torch.cuda.stream(streams[j]):
            moe.moe_ffn_forward_host(x_host[j], G["Wg"], G["W1"], G["W3"], G["W2"], k, out_host[j], ws_h[j],
                                     bias=G["bias"], Ws1=G["Ws1"], Ws3=G["Ws3"], Ws2=G["Ws2"])

    for i in range(max(args.warmup, nstream)):
        e2e_step(i)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for st in streams:
        st.wait_event(ev0)
    for i in range(K2):
        e2e_step(i)
    for st in streams:
        torch.cuda.current_stream().wait_stream(st)
    ev1.record()
    torch.cuda.synchronize()
    e2e = reduce_max(ev0.elapsed_time(ev1) / K2, dev)
    for j in range(1, nstream):  # every pipeline computed the same layer
        assert torch.equal(out_host[0], out_host[j])

    pk, pk_kind = peaks()
    st_mean = stage_ms
    sb = stage_bytes(w)
    fl = active_flops(w)
    tokens_s = T * world / (ms / 1e3)
    w1w3_s = st_mean["w1w3"] / 1e3
    achieved = w1w3_flops_per_launch(w) / w1w3_s / 1e12
    traffic = ncu_traffic(w1w3_kernel_name(w))
    hbm_stages = st_mean["route"] + st_mean["permute"] + st_mean["combine"]
    hbm_bytes = sb["route"] + sb["permute"] + sb["combine"]

    # ---- the other synthetic workloads, one GPU only (each timed like the headline) ----
    per_workload = None
    if world == 1 and not args.no_per_workload:
        del ws_h, x_host, out_host
        others = [n for n in inputs.WORKLOAD_ORDER if n != w.name]
        per_workload = measure_other_workloads(others, args, dev, moe, flush_l2, pk)
        per_workload[w.name] = {"see": "the headline keys of this line",
                                "roofline": roofline_place(w, ms, pk)}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        tps, n, runs, secs = time_oracle(L, w)
        cpu = {"value": tps, "unit": "tokens/s", "cores": host_cores(), "kind": "oracle",
               "sample": f"{runs} runs of the first {n} of {w.T} tokens through the whole layer "
                         f"({secs:.1f} s of fp64 numpy oracle)",
               "near_tie_tokens": near_tie_tokens(L, w)}
    line = {
        "metric": METRIC, "value": tokens_s, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": line_config(w, world),
        "ms_per_step_median": float(np.median(step_ms)),
        "active_tflops": fl * world / (ms / 1e3) / 1e12,
        "frac_of_bf16_peak": fl / (ms / 1e3) / 1e12 / pk["bf16_tflops"],
        "frac_of_datasheet_bf16_dense": fl / (ms / 1e3) / 1e12 / DATASHEET_BF16_DENSE_TFLOPS,
        "stage_ms": st_mean,
        "stage_ms_note": f"{KB} extra steps with an event at every stage boundary (serialised launches)",
        "roofline": {"bound": "tensor", "kernel": w1w3_kernel_name(w) + " (W1||W3 + SiLU*mul)",
                     "achieved": achieved, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / pk["bf16_tflops"], "traffic": traffic,
                     "peak_kind": f"{pk_kind} bf16 burst"},
        "hbm_stages": {"kernels": "route + permute + combine", "bytes": hbm_bytes, "ms": hbm_stages,
                       "achieved_gbs": hbm_bytes / (hbm_stages / 1e3) / 1e9,
                       "frac": hbm_bytes / (hbm_stages / 1e3) / 1e9 / pk["hbm_gbs"]},
        "read_reference": {"what": "event-timed after the same L2 flush: torch's float32 sum over x's bytes "
                                   "(a plain library read of T*D*2 bytes) and an empty kernel launch",
                           "x_bytes": T * D * 2, "torch_sum_x_ms": ref_ms["torch_sum_x"],
                           "empty_launch_ms": ref_ms["empty_launch"], "route_stage_ms": st_mean["route"]},
        "e2e": {"value": T * world / (e2e / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": T * D * 2, "d2h_bytes_per_step": T * D * 2,
                "ms_per_step": e2e, "steps": K2, "pipelining": f"{nstream} streams, copies overlap compute"},
        "graph": {"ms_per_step": graph_ms, "value": T * world / (graph_ms / 1e3), "unit": "tokens/s",
                  "note": "the same step captured once in a CUDA graph and replayed"},
        "gpu_launches": int(n_launch),
        "clocks": clocks,
        "wall_s_timed_loop": wall,
        "cpu_baseline": cpu,
        "per_workload": per_workload,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
