#!/usr/bin/env python
"""Benchmark: weight-stream GB/s of the low-bit GEMV/GEMM path on GB300.

Headline workload (one "step"): decode through one 4B-class dense decoder layer -- the seven
INT4 group-128 W4A16 projections (q, k, v, o, gate, up with K=2560; down with K=9728) at
M=1, 50,012,160 algorithmic weight bytes per step.  Every step reads a different copy of the
layer's packed weights (copies totalling more than 4x the L2 size), so timed weights come
from HBM.  Steps are replayed from per-copy CUDA graphs and timed with CUDA events.

Also reported under "rows": the M=16 verify GEMM over the same layer and its batch sweep,
binary-plane GEMV/GEMM, and the LM-head argmax+verify over 248,320 and 32,768 rows.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-rows]

N > 1 runs one independent replica per GPU (the path has no cross-GPU exchange); the value is
the whole-job throughput (all ranks' bytes / the slowest rank's time).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "weight-stream GB/s (% of HBM peak) and tok/s, low-bit GEMV/GEMM at M=1 and M=16"
LAYER_BYTES = 50_012_160


# ----------------------------------------------------------------------------- helpers

def algorithmic_int4_bytes(N, K):
    return N * K // 2 + N * (K // 128) * 2


def algorithmic_binplane_bytes(P, N, K):
    return P * N * K // 8 + P * N * (K // 128) * 2


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def reduce_max(value: float, world: int) -> float:
    """Max of a float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, seconds_per_rank: float, world: int) -> tuple:
    """(aggregate units/s, slowest rank's seconds): every rank processes the same units."""
    slowest = reduce_max(seconds_per_rank, world)
    return units_per_rank * world / slowest, slowest


class ClockSampler:
    """nvidia-smi clock/throttle sampling around a timed region."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            time.sleep(0.4)
        except OSError:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.count(",") >= 9]
        os.unlink(self.f.name)
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[2]))
                smax.append(float(r[3]))
                power.append(float(r[4]))
            except ValueError:
                continue
            for nm, v in zip(names, r[6:10]):
                if v.strip().lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s in sm if s >= 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------------------- GPU arm

def dev(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    return (t.view(dtype) if dtype is not None else t).cuda()


def bf16_dev(bits):
    import torch
    return dev(bits.view(np.int16), torch.bfloat16)


def f16_dev(bits):
    import torch
    return dev(bits.view(np.int16), torch.float16)


class Layer:
    """Packed INT4 projections of one 4B-class layer, replicated into C device copies."""

    def __init__(self, lb, torch, copies: int, M: int, seed: int):
        self.M = M
        self.shapes = [(k, n) for _, k, n in synth.LAYER_4B]
        self.packed = [[None] * len(self.shapes) for _ in range(copies)]
        self.X, self.Y = [], []
        for j, (K, N) in enumerate(self.shapes):
            codes, scales, x = synth.int4_problem(seed, M, N, K, j)
            p = torch.empty(lb.lowbit_int4_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
            lb.lowbit_pack_int4(dev(codes), f16_dev(scales), N, K, p)
            for c in range(copies):
                self.packed[c][j] = p if c == 0 else p.clone()
            self.X.append(bf16_dev(x))
            self.Y.append(torch.empty((M, N), dtype=torch.bfloat16, device="cuda"))
        self.bytes = sum(algorithmic_int4_bytes(N, K) for K, N in self.shapes)

    def step(self, lb, c, M=None):
        M = M or self.M
        for j, (K, N) in enumerate(self.shapes):
            lb.lowbit_gemm_int4(self.X[j], self.packed[c][j], M, N, K, self.Y[j])


def capture(torch, fn, n):
    """One CUDA graph per rotation slot i (fn(i) enqueues one step)."""
    graphs = []
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(n):
            fn(i)                      # eager warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for i in range(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            fn(i)
        graphs.append(g)
    torch.cuda.synchronize()
    return graphs


def time_graphs(torch, graphs, steps, warmup, world=1):
    for i in range(warmup):
        graphs[i % len(graphs)].replay()
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for i in range(steps):
        graphs[i % len(graphs)].replay()
    e1.record(st)
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    return e0.elapsed_time(e1) / 1e3


def copies_for(bytes_per_copy, l2_bytes, factor=4):
    return max(2, math.ceil(factor * l2_bytes / max(1, bytes_per_copy)))


def measure_rows(lb, torch, peak, l2, budget_s=1.0):
    """Secondary rows: M=16 verify GEMM + batch sweep, binary planes, LM head."""
    rows = {}

    def run(name, bytes_per_call, calls_per_step, fns, tokens_per_step, kernel):  # noqa: E306
        graphs = capture(torch, fns, fns.n)
        t1 = time_graphs(torch, graphs, 3, 2)
        steps = max(10, int(budget_s / max(t1 / 3, 1e-6)))
        secs = time_graphs(torch, graphs, steps, 5)
        per = secs / steps
        gbs = bytes_per_call * calls_per_step / per / 1e9
        rows[name] = {"us_per_step": round(per * 1e6, 3), "GB_s": round(gbs, 1),
                      "frac_of_hbm_peak": round(gbs / peak, 4), "tok_s": round(tokens_per_step / per, 1),
                      "kernel": kernel, "steps": steps}
        del graphs

    class Fns:
        def __init__(self, n, f):
            self.n, self.f = n, f

        def __call__(self, i):
            self.f(i)

    # config 2 and the batch sweep over the same layer
    layer = Layer(lb, torch, copies_for(LAYER_BYTES, l2), 32, seed=2)
    for M in synth.M_SWEEP:
        run(f"int4_layer_M{M}", layer.bytes, 1,
            Fns(len(layer.packed), lambda i, M=M: layer.step(lb, i, M)), M,
            "int4_gemv" if M == 1 else "int4_gemm")
    del layer
    torch.cuda.empty_cache()

    # config 3: binary planes
    for (K, N) in synth.BINPLANE_SHAPES:
        for P in synth.BINPLANE_PLANES:
            bits, alpha, x = synth.binplane_problem(3, P, 16, N, K)
            p0 = torch.empty(lb.lowbit_binplane_packed_bytes(P, N, K), dtype=torch.uint8, device="cuda")
            lb.lowbit_pack_binplane(dev(bits), f16_dev(alpha), P, N, K, p0)
            nb = algorithmic_binplane_bytes(P, N, K)
            C = copies_for(nb, l2)
            packs = [p0] + [p0.clone() for _ in range(C - 1)]
            X = bf16_dev(x)
            for M in (1, 16):
                Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
                run(f"binplane_K{K}_N{N}_P{P}_M{M}", nb, 1,
                    Fns(C, lambda i, M=M, Y=Y: lb.lowbit_gemm_binplane(X, packs[i], P, M, N, K, Y)),
                    M, "binplane")
            del packs, p0
            torch.cuda.empty_cache()

    # config 4: LM head verify
    M, K = synth.VERIFY_BLOCK, synth.HEAD_K
    for N in synth.HEAD_ROWS:
        codes, scales, h = synth.int4_problem(4, M, N, K)
        p0 = torch.empty(lb.lowbit_int4_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
        lb.lowbit_pack_int4(dev(codes), f16_dev(scales), N, K, p0)
        del codes
        nb = algorithmic_int4_bytes(N, K)
        C = copies_for(nb, l2, 2)
        packs = [p0] + [p0.clone() for _ in range(C - 1)]
        H = bf16_dev(h)
        drafts = dev(np.arange(M - 1, dtype=np.int32))
        a = torch.empty(M, dtype=torch.int32, device="cuda")
        n1 = torch.empty(1, dtype=torch.int32, device="cuda")
        b1 = torch.empty(1, dtype=torch.int32, device="cuda")
        ws = torch.zeros(lb.lmhead_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
        run(f"lmhead_N{N}_M{M}", nb, 1,
            Fns(C, lambda i: lb.lmhead_argmax_verify(H, packs[i], M, N, K, drafts, a, n1, b1, ws)),
            M, "lmhead")
        del packs, p0
        torch.cuda.empty_cache()
    return rows


def cpu_baseline_oracle(budget_s=10.0, rows_fraction=1.0):
    """The oracle (fp64 dequant + multiply) on the layer's seven projections at M=1."""
    from oracle import int4 as oint4
    probs = []
    for j, (_, K, N) in enumerate(synth.LAYER_4B):
        codes, scales, x = synth.int4_problem(1, 1, N, K, j)
        n = max(1, int(round(N * rows_fraction)))
        probs.append((codes[:n], scales[:n], x, algorithmic_int4_bytes(n, K)))
    nbytes = sum(p[3] for p in probs)
    t0 = time.perf_counter()
    reps = 0
    while True:
        for codes, scales, x, _ in probs:
            oint4.gemm(x, codes, scales)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    secs = time.perf_counter() - t0
    return nbytes * reps / secs / 1e9, reps, nbytes, secs


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    import bit_weight_gemv_gb300 as lb

    peak, peak_kind = read_peaks()
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    C = copies_for(LAYER_BYTES, l2)
    layer = Layer(lb, torch, C, 1, seed=1)
    assert layer.bytes == LAYER_BYTES
    graphs = capture(torch, lambda i: layer.step(lb, i), C)

    sampler = ClockSampler(local)
    sampler.start()
    secs = time_graphs(torch, graphs, args.steps, args.warmup, world)
    clocks = sampler.stop()
    units = LAYER_BYTES * args.steps
    rate, slowest = whole_job_rate(units, secs, world)
    value = rate / 1e9
    per_rank_gbs = units / secs / 1e9
    launches = 7 * args.steps

    # e2e through the public API with host buffers: H2D of X, 7 GEMVs, D2H of Y per step
    Xh = [x.cpu().pin_memory() for x in layer.X]
    Yh = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for y in layer.Y]
    h2d = sum(x.numel() * 2 for x in Xh)
    d2h = sum(y.numel() * 2 for y in Yh)
    e2e_steps = max(20, min(args.steps, 2000))

    def e2e_step(i):
        for j, (K, N) in enumerate(layer.shapes):
            layer.X[j].copy_(Xh[j], non_blocking=True)
            lb.lowbit_gemm_int4(layer.X[j], layer.packed[i % C][j], 1, N, K, layer.Y[j])
            Yh[j].copy_(layer.Y[j], non_blocking=True)

    for i in range(5):
        e2e_step(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_secs = time.perf_counter() - t0
    e2e_rate, _ = whole_job_rate(LAYER_BYTES * e2e_steps, e2e_secs, world)

    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        with open(tpath) as f:
            tj = json.load(f)
        ent = tj.get("int4_gemv_kernel@decode_layer")
        if ent and ent.get("src_sha") == _src_sha("int4_cc.cu"):
            traffic = ent.get("bytes_per_launch")

    rows = {}
    if not args.no_rows and rank == 0:
        rows = measure_rows(lb, torch, peak, l2)

    cpu = None
    if rank == 0:
        gbs, reps, nbytes, csecs = cpu_baseline_oracle(args.cpu_budget)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{reps} passes of the oracle (numpy fp64 dequant + multiply) over the "
                         f"seven M=1 projections of one layer ({nbytes} algorithmic bytes each), "
                         f"{csecs:.1f} s"}

    if rank == 0:
        out = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(slowest / args.steps * 1e3, 6), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "decode W4A16 GEMV over one 4B-class layer: q,k,v,o,gate,up "
                                   "(K=2560) and down (K=9728), INT4 group 128, M=1",
                       "M": 1, "weight_bytes_per_step": LAYER_BYTES, "rotating_copies": C,
                       "l2_policy": f"inputs larger than L2: {C} rotating weight copies, "
                                    f"{C * LAYER_BYTES / 1e6:.0f} MB vs L2 {l2 / 1e6:.0f} MB",
                       "replay": "per-copy CUDA graphs"},
            "tok_s": round(args.steps * world / slowest, 1),
            "roofline": {"bound": "hbm", "achieved": round(per_rank_gbs, 2), "peak": peak,
                         "unit": "GB/s", "frac": round(per_rank_gbs / peak, 4),
                         "peak_source": peak_kind, "traffic": traffic,
                         "kernel": "int4_gemv_kernel",
                         "algorithmic_bytes_per_launch": LAYER_BYTES / 7},
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_rate / 1e9, 2), "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "note": "eager API calls per step with pinned host X/Y, 7 projections"},
            "gpu_launches": launches,
            "clocks": clocks,
            "rows": rows,
        }
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def _src_sha(name):
    import hashlib
    p = os.path.join(ROOT, "bit_weight_gemv_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


# ----------------------------------------------------------------------------- reference arm

def run_reference(args):
    """The CPU oracle as it stands, on a bounded sample of each step's layer."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    # calibrate: one full-layer pass, then choose a row fraction so the run takes ~90 s
    gbs_full, _, nbytes_full, secs_full = cpu_baseline_oracle(budget_s=0.0)
    per_step_budget = 90.0 / max(1, args.steps + args.warmup)
    frac = min(1.0, per_step_budget / max(secs_full, 1e-9))
    from oracle import int4 as oint4
    probs = []
    for j, (_, K, N) in enumerate(synth.LAYER_4B):
        codes, scales, x = synth.int4_problem(1, 1, N, K, j)
        n = max(1, int(round(N * frac)))
        probs.append((codes[:n], scales[:n], x, algorithmic_int4_bytes(n, K)))
    nbytes = sum(p[3] for p in probs)
    for _ in range(args.warmup):
        for codes, scales, x, _ in probs:
            oint4.gemm(x, codes, scales)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for codes, scales, x, _ in probs:
            oint4.gemm(x, codes, scales)
    secs = time.perf_counter() - t0
    value = nbytes * args.steps / secs / 1e9
    sample = (f"each step: the oracle over {frac:.4%} of the rows of each of the seven M=1 "
              f"projections ({nbytes} algorithmic bytes)")
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(secs / args.steps * 1e3, 4), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": "decode W4A16 GEMV over one 4B-class layer: q,k,v,o,gate,up "
                                  "(K=2560) and down (K=9728), INT4 group 128, M=1", "M": 1},
           "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": os.cpu_count(),
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-rows", action="store_true", help="skip the secondary rows")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle timing")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
