#!/usr/bin/env python
"""Benchmark: weight-stream GB/s of the low-bit GEMV/GEMM path on GB300.

Headline workload (one "step"): decode through one 4B-class dense decoder layer -- the seven
INT4 group-128 W4A16 projections (q, k, v, o, gate, up with K=2560; down with K=9728) at
M=1, 50,012,160 algorithmic weight bytes per step, issued the way a decoder's data
dependencies allow: lowbit_gemm_int4_grouped over (q, k, v), then o, then (gate, up), then
down -- four launches.  Every step reads a different copy of the layer's packed weights
(copies totalling more than 4x the L2 size), so timed weights come from HBM.  Steps are
replayed from CUDA graphs (one per rotation of the weight copies) and timed with CUDA events.

Also reported under "rows": the same layer as seven single-matrix calls ("decode") and as one
grouped call ("decode_all"), the M=16 verify GEMM over the same layer and its batch sweep,
binary-plane GEMV/GEMM, the deployed ShiftAdd format (u8 scale codes, "sa_m1"/"sa_m16"), the
248,320-row vocabulary head as one M=1 GEMV ("head_gemv"), the trimmed NVFP4 and Q8 draft heads
with their id-mapped argmax ("draft_m1"/"draft_m16", "draft_q8_m1"/"draft_q8_m16"), and the
LM-head argmax+verify over 248,320 and 32,768 rows.

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
DEFAULT_WORKLOAD_DESC = ("decode W4A16 GEMV over one 4B-class layer, M=1, grouped as a decoder's "
                         "dependencies allow: (q,k,v), (o), (gate,up), (down), one launch each")


# ----------------------------------------------------------------------------- helpers

def algorithmic_int4_bytes(N, K):
    return N * K // 2 + N * (K // 128) * 2


def algorithmic_binplane_bytes(P, N, K):
    return P * N * K // 8 + P * N * (K // 128) * 2


def algorithmic_sa_bytes(P, G, N, K):
    """Sign bits, u8 scale codes and one fp16 d per 256 inputs."""
    return P * N * K // 8 + P * N * (K // G) + N * (K // 256) * 2


def algorithmic_q8_bytes(N, K):
    """int8 codes and one fp16 scale per 32 inputs."""
    return N * K + N * (K // 32) * 2


def algorithmic_nvfp4_bytes(N, K):
    """E2M1 codes and one E4M3 scale per 16 inputs."""
    return N * K // 2 + N * K // 16


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def read_tensor_peak():
    """bf16 dense tensor peak in TFLOP/s for a kernel timed alone (burst), and its source."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def step_stats(torch, rep, steps, repeats=20):
    """Per-step device time over `repeats` separately timed runs of steps // repeats steps
    each (after the main measurement): median, p10 and p90 in microseconds."""
    each = max(1, steps // repeats)
    ts = []
    for r in range(repeats):  # the rotation continues, so no repeat re-reads an L2-resident copy
        ts.append(time_graphs(torch, rep, each, 0, start=r * each) / each * 1e6)
    ts.sort()
    q = lambda f: ts[min(len(ts) - 1, int(round(f * (len(ts) - 1))))]
    return {"median_us": round(q(0.5), 3), "p10_us": round(q(0.1), 3), "p90_us": round(q(0.9), 3),
            "repeats": repeats, "steps_each": each}


def cold_step_us(torch, rep, l2_bytes):
    """One step right after L2 has been overwritten (a buffer twice its size), timed alone."""
    flush = torch.empty(2 * l2_bytes, dtype=torch.uint8, device="cuda")
    flush.fill_(1)
    torch.cuda.synchronize()
    us = time_graphs(torch, rep, 1, 0) * 1e6
    del flush
    return round(us, 3)

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


class Workload:
    """A timed step: a list of calls over one of C rotating device copies of the weights.

    name, description, M, weight bytes per step, tokens per step, launches per step, the
    dominant kernel's name, and C (copies) so that C * bytes >= 4x L2."""

    def __init__(self, name, desc, kernel):
        self.name, self.desc, self.kernel = name, desc, kernel
        self.calls = []          # per copy: list of zero-arg callables
        self.bytes = 0
        self.tokens = 0
        self.launches = 0
        self.M = 0
        self.weights = 0         # weight elements per step (N*K summed), for tensor flops
        self.host_io = None      # (inputs on device, outputs on device) for the e2e leg

    def step(self, c):
        for f in self.calls[c % len(self.calls)]:
            f()


def _copies(p0, n, torch):
    return [p0] + [p0.clone() for _ in range(n - 1)]


# Launch groupings of the layer's seven projections (q, k, v, o, gate, up, down):
#   None   : one lowbit_gemm_int4 call per projection (7 launches);
#   "deps" : what a decoder's data dependencies allow, one lowbit_gemm_int4_grouped call per
#            set -- (q, k, v) read the same input, o follows attention, (gate, up) share the
#            post-attention input, down follows the activation -- 4 launches;
#   "all"  : all seven in one grouped call (1 launch).
LAYER_GROUPS = {"deps": ((0, 1, 2), (3,), (4, 5), (6,)), "all": ((0, 1, 2, 3, 4, 5, 6),)}


def build_int4_layer(lb, torch, l2, M, path, seed, name, desc, grouping=None):
    if grouping is not None and path == 1 and M > 4:
        path = 0  # grouped calls have no CUDA-core kernel above the streaming kernel's 4 rows
    w = Workload(name, desc, "int4_stream_kernel" if ((M <= 2 and path == 0) or (M <= 4 and path == 1))
                 else {1: "int4_gemm_cc_kernel", 2: "tc_gemm_kernel"}.get(path, "int4_mma_kernel"))
    shapes = [(k, n) for _, k, n in synth.LAYER_4B]
    w.bytes = sum(algorithmic_int4_bytes(N, K) for K, N in shapes)
    w.weights = sum(N * K for K, N in shapes)
    C = copies_for(w.bytes, l2)
    # one device buffer for all activations and one for all outputs (16-byte aligned views),
    # so an end-to-end step moves them with one copy each way
    xoff = np.cumsum([0] + [M * K for K, _ in shapes])
    yoff = np.cumsum([0] + [M * N for _, N in shapes])
    Xflat = torch.empty(int(xoff[-1]), dtype=torch.bfloat16, device="cuda")
    Yflat = torch.empty(int(yoff[-1]), dtype=torch.bfloat16, device="cuda")
    packs, X, Y = [], [], []
    for j, (K, N) in enumerate(shapes):
        codes, scales, x = synth.int4_problem(seed, M, N, K, j)
        p = torch.empty(lb.lowbit_int4_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
        lb.lowbit_pack_int4(dev(codes), f16_dev(scales), N, K, p)
        packs.append(_copies(p, C, torch))
        X.append(Xflat[int(xoff[j]):int(xoff[j + 1])].view(M, K))
        X[-1].copy_(bf16_dev(x))
        Y.append(Yflat[int(yoff[j]):int(yoff[j + 1])].view(M, N))
    if grouping is None:
        for c in range(C):
            w.calls.append([(lambda j=j, K=K, N=N, c=c: lb.lowbit_gemm_int4_path(
                X[j], packs[j][c], M, N, K, Y[j], path)) for j, (K, N) in enumerate(shapes)])
        w.launches = len(shapes)
    else:
        groups = LAYER_GROUPS[grouping]
        for c in range(C):
            w.calls.append([(lambda grp=grp, c=c: lb.lowbit_gemm_int4_grouped_path(
                [(X[j], packs[j][c], shapes[j][1], shapes[j][0], Y[j]) for j in grp], M, path))
                for grp in groups])
        w.launches = len(groups)
    w.M, w.tokens = M, M
    w.host_io = (Xflat, Yflat)
    return w


def build_binplane(lb, torch, l2, M, path, name, desc):
    w = Workload(name, desc, "bp_stream_kernel" if (M == 1 and path in (0, 1))
                 else ("tc_gemm_kernel" if path == 2 else
                       ("binplane_cc_kernel" if path == 1 else "bp_mma_kernel")))
    mats = []
    for si, (K, N) in enumerate(synth.BINPLANE_SHAPES):
        for P in synth.BINPLANE_PLANES:
            bits, alpha, x = synth.binplane_problem(3, P, M, N, K, si)
            p = torch.empty(lb.lowbit_binplane_packed_bytes(P, N, K), dtype=torch.uint8, device="cuda")
            lb.lowbit_pack_binplane(dev(bits), f16_dev(alpha), P, N, K, p)
            mats.append((P, K, N, p, bf16_dev(x), torch.empty((M, N), dtype=torch.bfloat16, device="cuda")))
            w.bytes += algorithmic_binplane_bytes(P, N, K)
            w.weights += N * K
    C = copies_for(w.bytes, l2)
    copies = [_copies(m[3], C, torch) for m in mats]
    for c in range(C):
        w.calls.append([(lambda i=i, c=c: lb.lowbit_gemm_binplane_path(
            mats[i][4], copies[i][c], mats[i][0], M, mats[i][2], mats[i][1], mats[i][5], path))
            for i in range(len(mats))])
    w.M, w.tokens, w.launches = M, M, len(mats)
    return w


def build_sa(lb, torch, l2, M, name, desc, path=0):
    w = Workload(name, desc, "sa_stream_kernel" if M == 1 else
                 {1: "binplane_cc_kernel", 2: "tc_gemm_kernel"}.get(path, "sa_mma_kernel"))
    mats = []
    for si, (K, N) in enumerate(synth.SA_SHAPES):
        for P, G in synth.SA_TYPES:
            bits, codes, d, x = synth.sa_problem(3, P, G, M, N, K, si)
            p = torch.empty(lb.lowbit_sa_packed_bytes(P, G, N, K), dtype=torch.uint8, device="cuda")
            lb.lowbit_pack_sa(dev(bits), dev(codes), f16_dev(d), P, G, N, K, p)
            mats.append((P, G, K, N, p, bf16_dev(x), torch.empty((M, N), dtype=torch.bfloat16, device="cuda")))
            w.bytes += algorithmic_sa_bytes(P, G, N, K)
            w.weights += N * K
    C = copies_for(w.bytes, l2)
    copies = [_copies(m[4], C, torch) for m in mats]
    for c in range(C):
        w.calls.append([(lambda i=i, c=c: lb.lowbit_gemm_sa_path(
            mats[i][5], copies[i][c], mats[i][0], mats[i][1], M, mats[i][3], mats[i][2], mats[i][6],
            path)) for i in range(len(mats))])
    w.M, w.tokens, w.launches = M, M, len(mats)
    return w


def build_draft_head(lb, torch, l2, M, name, desc):
    """The trimmed NVFP4 draft head: argmax over its rows, mapped to full-vocabulary ids."""
    N, K = synth.DRAFT_ROWS, synth.HEAD_K
    w = Workload(name, desc, "nvfp4_stream_kernel" if M == 1 else "tc_gemm_kernel")
    codes, scales, g, ids, h = synth.nvfp4_problem(4, M, N, K)
    p = torch.empty(lb.lowbit_nvfp4_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    lb.lowbit_pack_nvfp4(dev(codes), dev(scales), g, N, K, p)
    w.bytes = algorithmic_nvfp4_bytes(N, K)
    w.weights = N * K
    packs = _copies(p, copies_for(w.bytes, l2), torch)
    H, idm = bf16_dev(h), dev(ids)
    out = torch.empty(M, dtype=torch.int32, device="cuda")
    ws = torch.zeros(lb.lmhead_workspace_bytes(2, N, K), dtype=torch.uint8, device="cuda")
    for c in range(len(packs)):
        w.calls.append([lambda c=c: lb.lowbit_draft_argmax(H, packs[c], M, N, K, idm, out, ws)])
    w.M, w.tokens, w.launches = M, M, 1
    return w


def build_q8_head(lb, torch, l2, M, name, desc):
    """The trimmed head in Q8: argmax over its rows, mapped to full-vocabulary ids."""
    N, K = synth.DRAFT_ROWS, synth.HEAD_K
    w = Workload(name, desc, "q8_stream_kernel" if M == 1 else "q8_mma_kernel")
    codes, scales, ids, h = synth.q8_problem(4, M, N, K)
    p = torch.empty(lb.lowbit_q8_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    lb.lowbit_pack_q8(dev(codes), f16_dev(scales), N, K, p)
    w.bytes = algorithmic_q8_bytes(N, K)
    w.weights = N * K
    packs = _copies(p, copies_for(w.bytes, l2), torch)
    H, idm = bf16_dev(h), dev(ids)
    out = torch.empty(M, dtype=torch.int32, device="cuda")
    ws = torch.zeros(lb.lmhead_workspace_bytes(2, N, K), dtype=torch.uint8, device="cuda")
    for c in range(len(packs)):
        w.calls.append([lambda c=c: lb.lowbit_draft_argmax_q8(H, packs[c], M, N, K, idm, out, ws)])
    w.M, w.tokens, w.launches = M, M, 1
    return w


def build_lmhead(lb, torch, l2, N, path, name, desc):
    M, K = synth.VERIFY_BLOCK, synth.HEAD_K
    w = Workload(name, desc, {1: "int4_gemm_cc_kernel", 2: "tc_gemm_kernel"}.get(path, "int4_mma_kernel"))
    codes, scales, h = synth.int4_problem(4, M, N, K)
    p = torch.empty(lb.lowbit_int4_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    lb.lowbit_pack_int4(dev(codes), f16_dev(scales), N, K, p)
    del codes
    w.bytes = algorithmic_int4_bytes(N, K)
    w.weights = N * K
    C = copies_for(w.bytes, l2, 2)
    packs = _copies(p, C, torch)
    H = bf16_dev(h)
    drafts = dev(np.arange(M - 1, dtype=np.int32))
    a = torch.empty(M, dtype=torch.int32, device="cuda")
    n1 = torch.empty(1, dtype=torch.int32, device="cuda")
    b1 = torch.empty(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(lb.lmhead_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    for c in range(C):
        w.calls.append([lambda c=c: lb.lmhead_argmax_verify_path(H, packs[c], M, N, K, drafts, a, n1,
                                                                 b1, ws, path)])
    w.M, w.tokens, w.launches = M, M, 1
    return w


def build_head_gemv(lb, torch, l2, path, name, desc):
    """One large INT4 matrix at M=1: the full vocabulary head's logits for one token."""
    N, K = synth.HEAD_ROWS[0], synth.HEAD_K
    w = Workload(name, desc, "int4_stream_kernel" if path != 2 else "tc_gemm_kernel")
    codes, scales, x = synth.int4_problem(4, 1, N, K, 1)
    p = torch.empty(lb.lowbit_int4_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    lb.lowbit_pack_int4(dev(codes), f16_dev(scales), N, K, p)
    del codes
    w.bytes = algorithmic_int4_bytes(N, K)
    w.weights = N * K
    packs = _copies(p, copies_for(w.bytes, l2, 2), torch)
    X, Y = bf16_dev(x), torch.empty((1, N), dtype=torch.bfloat16, device="cuda")
    for c in range(len(packs)):
        w.calls.append([lambda c=c: lb.lowbit_gemm_int4_path(X, packs[c], 1, N, K, Y, path)])
    w.M, w.tokens, w.launches = 1, 1, 1
    return w


def build_workload(lb, torch, l2, name, path):
    if name == "decode":
        return build_int4_layer(lb, torch, l2, 1, path, 1, name,
                                "decode W4A16 GEMV over one 4B-class layer: q,k,v,o,gate,up (K=2560) "
                                "and down (K=9728), INT4 group 128, M=1")
    if name in ("decode_deps", "decode_all"):
        grouping = name.split("_")[1]
        desc = (DEFAULT_WORKLOAD_DESC if grouping == "deps" else
                "decode W4A16 GEMV over one 4B-class layer, M=1, all seven in one grouped launch")
        return build_int4_layer(lb, torch, l2, 1, path, 1, name, desc, grouping=grouping)
    if name in ("verify_deps", "verify_all"):
        grouping = name.split("_")[1]
        how = ("grouped as a decoder's dependencies allow: (q,k,v), (o), (gate,up), (down), "
               "one launch each" if grouping == "deps" else "all seven in one grouped launch")
        return build_int4_layer(lb, torch, l2, 16, path, 2, name,
                                "speculative-verify skinny GEMM over the same 4B-class layer, M=16, "
                                + how, grouping=grouping)
    if name == "verify":
        return build_int4_layer(lb, torch, l2, 16, path, 2, name,
                                "speculative-verify skinny GEMM over the same 4B-class layer, M=16")
    if name.startswith("verify_m"):
        M = int(name[len("verify_m"):])
        return build_int4_layer(lb, torch, l2, M, path, 2, name,
                                f"batch sweep: the 4B-class layer at M={M}")
    if name == "tiny":
        w = Workload(name, "tiny INT4 GEMV K=512 N=256 M=1", "int4_stream_kernel")
        codes, scales, x = synth.int4_problem(0, 1, 256, 512)
        p = torch.empty(lb.lowbit_int4_packed_bytes(256, 512), dtype=torch.uint8, device="cuda")
        lb.lowbit_pack_int4(dev(codes), f16_dev(scales), 256, 512, p)
        X, Y = bf16_dev(x), torch.empty((1, 256), dtype=torch.bfloat16, device="cuda")
        w.calls = [[lambda: lb.lowbit_gemm_int4_path(X, p, 1, 256, 512, Y, path)]]
        w.bytes, w.M, w.tokens, w.launches = algorithmic_int4_bytes(256, 512), 1, 1, 1
        return w
    if name in ("binplane_m1", "binplane_m16"):
        M = 1 if name == "binplane_m1" else 16
        return build_binplane(lb, torch, l2, M, path, name,
                              f"binary-plane GEMM: (K,N) in {{(4096,12288),(12288,4096)}} x P in {{3,4}}, "
                              f"M={M}, group 128")
    if name in ("sa_m1", "sa_m16"):
        M = 1 if name == "sa_m1" else 16
        types = ", ".join(f"sa{P}{'' if G == 64 else '_' + str(G)}" for P, G in synth.SA_TYPES)
        return build_sa(lb, torch, l2, M, name,
                        f"deployed ShiftAdd format ({types}: u8 scale codes, fp16 d per 256 inputs): "
                        f"(K,N) in {{(4096,12288),(12288,4096)}}, M={M}", path)
    if name in ("draft_m1", "draft_m16"):
        M = 1 if name == "draft_m1" else 16
        return build_draft_head(lb, torch, l2, M, name,
                                f"trimmed NVFP4 draft head: {synth.DRAFT_ROWS} rows x K={synth.HEAD_K}, "
                                f"M={M}, fused argmax mapped to full-vocabulary ids")
    if name in ("draft_q8_m1", "draft_q8_m16"):
        M = 1 if name == "draft_q8_m1" else 16
        return build_q8_head(lb, torch, l2, M, name,
                             f"trimmed Q8 draft head (int8, fp16 scale per 32): {synth.DRAFT_ROWS} rows x "
                             f"K={synth.HEAD_K}, M={M}, fused argmax mapped to full-vocabulary ids")
    if name == "head_gemv":
        return build_head_gemv(lb, torch, l2, path, name,
                               f"INT4 GEMV at M=1 over the {synth.HEAD_ROWS[0]}-row vocabulary head, "
                               f"K={synth.HEAD_K}, group 128 (one 524 MB matrix)")
    if name in ("lmhead_full", "lmhead_trim"):
        N = synth.HEAD_ROWS[0] if name == "lmhead_full" else synth.HEAD_ROWS[1]
        return build_lmhead(lb, torch, l2, N, path, name,
                            f"LM-head verify: M=16, K=4096, INT4 head of N={N} rows, fused argmax + "
                            "greedy acceptance of 15 drafts")
    raise ValueError(name)


WORKLOADS = ("decode", "decode_deps", "decode_all", "verify", "verify_deps", "verify_all", "binplane_m1", "binplane_m16", "sa_m1", "sa_m16", "draft_m1", "draft_m16", "draft_q8_m1", "draft_q8_m16", "head_gemv", "lmhead_full", "lmhead_trim",
             "tiny") + tuple(f"verify_m{m}" for m in synth.M_SWEEP if m not in (16,))


class Replay:
    """CUDA graphs for a workload, captured ahead of any timed region.

    A run of `steps` steps starting at weight copy `start` is replayed from graphs covering
    exactly those steps: one graph when the run is short (up to `short` steps), otherwise a
    graph up to the next rotation boundary, whole-rotation graphs (n steps, one per weight
    copy) and a graph for the remainder.  Graphs are captured on first use and cached, so the
    host pays a handful of graph launches per timed run and the GPU sees the steps back to back."""

    def __init__(self, torch, step, n, short=512):
        self.torch, self.step, self.n, self.short = torch, step, n, short
        self.cache = {}

    def _graph(self, start, length):
        key = (start % self.n, length)
        g = self.cache.get(key)
        if g is None:
            torch = self.torch
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, capture_error_mode="thread_local"):
                for i in range(start, start + length):
                    self.step(i)
            torch.cuda.synchronize()
            self.cache[key] = g
        return g

    def plan(self, steps, start=0):
        """The graphs that replay steps start .. start + steps - 1 (captured now if needed)."""
        if steps <= 0:
            return []
        if steps <= self.short:
            return [self._graph(start, steps)]
        out, i = [], start
        head = min((-i) % self.n, steps)  # up to the next rotation boundary, or the whole run
        if head:
            out.append(self._graph(i, head))
            i += head
        full = (start + steps - i) // self.n
        out += [self._graph(0, self.n)] * full
        i += full * self.n
        if start + steps > i:
            out.append(self._graph(i, start + steps - i))
        return out

    def run(self, steps, start=0):
        for g in self.plan(steps, start):
            g.replay()
        return start + steps


def capture(torch, w, n):
    """Eager warm-up of every weight copy (outside any capture), then a graph replayer."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(n):
            w.step(i)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return Replay(torch, w.step, n)


def time_graphs(torch, rep, steps, warmup, world=1, start=0):
    """Device time of exactly `steps` steps after `warmup` untimed ones (CUDA events on the
    launching stream, barrier + synchronize on both sides).  Every graph either run replays is
    captured before the timed region starts."""
    warm = rep.plan(warmup, start)
    timed = rep.plan(steps, start + warmup)
    # a graph's first launch also uploads it to the device: launch every graph of the timed
    # run once beforehand (untimed), then the W warm-up steps
    for g in {id(g): g for g in timed}.values():
        g.replay()
    for g in warm:
        g.replay()
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for g in timed:
        g.replay()
    e1.record(st)
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    return e0.elapsed_time(e1) / 1e3


def copies_for(bytes_per_copy, l2_bytes, factor=4):
    return max(2, math.ceil(factor * l2_bytes / max(1, bytes_per_copy)))


def measure_rows(lb, torch, peak, l2, names, budget_s=0.5):
    """Secondary rows: every other workload, timed the same way (CUDA graphs, rotation), with
    the spread of 10 separately timed repeats and, at M >= 16, the fraction of the bf16 tensor
    peak (dense-equivalent 2*M*N*K flops)."""
    rows = {}
    tpeak, _ = read_tensor_peak()
    for name, path in names:
        w = build_workload(lb, torch, l2, name, path)
        graphs = capture(torch, w, len(w.calls))
        t1 = time_graphs(torch, graphs, 3, 2)
        steps = max(10, int(budget_s / max(t1 / 3, 1e-6)))
        secs = time_graphs(torch, graphs, steps, 5)
        per = secs / steps
        gbs = w.bytes / per / 1e9
        key = name if path == 0 else f"{name}@path{path}"
        rows[key] = {"us_per_step": round(per * 1e6, 3), "GB_s": round(gbs, 1),
                     "frac_of_hbm_peak": round(gbs / peak, 4), "tok_s": round(w.tokens / per, 1),
                     "kernel": w.kernel, "launches_per_step": w.launches, "steps": steps,
                     "weight_bytes_per_step": w.bytes,
                     "spread": step_stats(torch, graphs, max(10, steps // 2), repeats=10)}
        if w.M >= 16 and w.weights:
            tf = 2.0 * w.M * w.weights / per / 1e12
            rows[key]["tensor_tflops"] = round(tf, 2)
            rows[key]["frac_of_tensor_peak"] = round(tf / tpeak, 4)
        del graphs, w
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


THREAD_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def os_threads():
    """Threads of this process right now (Linux), or None."""
    try:
        return len(os.listdir("/proc/self/task"))
    except OSError:
        return None


def cpu_baseline_child(threads, budget_s):
    """Time the oracle in a fresh interpreter whose BLAS and OpenMP pools are limited to
    `threads` (the limit is read when numpy loads, so it needs its own process)."""
    env = dict(os.environ)
    for k in THREAD_ENV:
        env[k] = str(threads)
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-child",
                        "--cpu-budget", str(budget_s)], env=env, capture_output=True, text=True,
                       timeout=budget_s * 6 + 120)
    if r.returncode != 0:
        return None
    d = json.loads(r.stdout.strip().splitlines()[-1])
    d["threads_requested"] = threads
    return d


def cpu_baseline_two_modes(budget_s):
    """CPU baseline: the oracle with one thread and with every host core."""
    cores = os.cpu_count() or 1
    one = cpu_baseline_child(1, budget_s / 2)
    allc = cpu_baseline_child(cores, budget_s / 2)
    if allc is None:
        return None
    sample = (f"{allc['reps']} passes of the oracle (numpy fp64 dequant + multiply) over "
              f"{allc['row_fraction']:.2%} of the rows of each of the seven M=1 projections of one "
              f"layer ({allc['nbytes']} algorithmic bytes per pass), {allc['secs']:.1f} s")
    out = {"value": round(allc["gbs"], 4), "unit": "GB/s", "cores": allc["threads_requested"],
           "threads_seen": allc["threads_seen"], "kind": "oracle", "sample": sample,
           "thread_env": ",".join(THREAD_ENV)}
    if one is not None:
        out["one_thread"] = {"value": round(one["gbs"], 4), "unit": "GB/s", "cores": 1,
                             "threads_seen": one["threads_seen"],
                             "sample": f"{one['reps']} passes over {one['row_fraction']:.2%} of "
                                       f"the rows ({one['nbytes']} bytes per pass), {one['secs']:.1f} s"}
    return out


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
    w = build_workload(lb, torch, l2, args.workload, args.path)
    C = len(w.calls)
    graphs = capture(torch, w, C)

    sampler = ClockSampler(local)
    sampler.start()
    secs = time_graphs(torch, graphs, args.steps, args.warmup, world)
    clocks = sampler.stop()
    units = w.bytes * args.steps
    rate, slowest = whole_job_rate(units, secs, world)
    per_rank_gbs = units / secs / 1e9
    # outside the timed region: the spread of separately timed repeats, and one cold step
    spread = step_stats(torch, graphs, args.steps)
    cold = cold_step_us(torch, graphs, l2)
    del graphs

    # e2e through the public API with host buffers: every step copies the step's activations
    # in from pinned host memory (one copy), makes the step's library calls, and copies all
    # outputs back (one copy).  Timed on the host clock around graph replays of those steps,
    # the way a serving loop issues a decode step; the same steps issued eagerly from Python
    # are reported beside it as the host's issue rate.
    e2e = None
    if w.host_io is not None:
        Xd, Yd = w.host_io
        Xh = Xd.cpu().pin_memory()
        Yh = torch.empty(Yd.shape, dtype=Yd.dtype).pin_memory()
        h2d, d2h = Xh.numel() * Xh.element_size(), Yh.numel() * Yh.element_size()

        def e2e_step(i):
            Xd.copy_(Xh, non_blocking=True)
            w.step(i)
            Yh.copy_(Yd, non_blocking=True)

        e2e_rep = Replay(torch, e2e_step, C)
        e2e_steps = max(20, min(args.steps, 2000))
        timed = e2e_rep.plan(e2e_steps, 5)
        e2e_rep.run(5)
        torch.cuda.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        t0 = time.perf_counter()
        for g in timed:
            g.replay()
        torch.cuda.synchronize()
        e2e_secs = time.perf_counter() - t0
        e2e_rate, _ = whole_job_rate(w.bytes * e2e_steps, e2e_secs, world)
        for i in range(5):
            e2e_step(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            e2e_step(i)
        torch.cuda.synchronize()
        eager_rate, _ = whole_job_rate(w.bytes * e2e_steps, time.perf_counter() - t0, world)
        del e2e_rep
        e2e = {"value": round(e2e_rate / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "note": "host clock around graph replays of steps that copy the activations in "
                       "from pinned host memory, call the library, and copy the outputs out",
               "eager_value": round(eager_rate / 1e9, 2),
               "eager_note": "the same steps as eager Python calls (host issue rate)"}

    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        with open(tpath) as f:
            tj = json.load(f)
        ent = tj.get(f"{w.kernel}@{args.workload}")
        if ent and ent.get("src_sha") == _src_sha(ent.get("sources", ())):
            traffic = ent.get("bytes_per_launch")

    rows = {}
    if not args.no_rows and rank == 0:
        names = [(n, 0) for n in WORKLOADS if n not in (args.workload, "tiny")]
        names += [("decode", 2), ("binplane_m1", 1), ("binplane_m1", 2), ("verify_all", 2),
                  ("lmhead_full", 2), ("binplane_m16", 2), ("sa_m16", 2)]
        names = [nm for nm in names if nm != (args.workload, args.path)]
        rows = measure_rows(lb, torch, peak, l2, names)

    cpu = None
    if rank == 0 and args.cpu_budget > 0:
        cpu = cpu_baseline_two_modes(args.cpu_budget)

    if rank == 0:
        out = {
            "metric": METRIC, "value": round(rate / 1e9, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(slowest / args.steps * 1e3, 6), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.desc, "name": args.workload, "M": w.M,
                       "weight_bytes_per_step": w.bytes, "rotating_copies": C,
                       "l2_policy": f"inputs larger than L2: {C} rotating weight copies, "
                                    f"{C * w.bytes / 1e6:.0f} MB vs L2 {l2 / 1e6:.0f} MB",
                       "replay": "CUDA graphs covering exactly the timed steps, captured and "
                                 "launched once (untimed) before the warm-up steps",
                       "kernel_path": args.path, "arith": arith_note(w)},
            "tok_s": round(w.tokens * args.steps * world / slowest, 1),
            "roofline": {"bound": "hbm", "achieved": round(per_rank_gbs, 2), "peak": peak,
                         "unit": "GB/s", "frac": round(per_rank_gbs / peak, 4),
                         "peak_source": peak_kind, "traffic": traffic, "kernel": w.kernel,
                         "algorithmic_bytes_per_launch": w.bytes / w.launches,
                         "launches_per_step": w.launches},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": w.launches * args.steps,
            "clocks": clocks,
            "step_time_spread": spread,
            "cold_step_us": cold,
            "rows": rows,
        }
        if w.M >= 16 and w.weights:
            tpeak, tkind = read_tensor_peak()
            tf = 2.0 * w.M * w.weights * args.steps / secs / 1e12
            out["tensor"] = {"tflops": round(tf, 2), "peak": tpeak, "peak_source": tkind,
                             "frac": round(tf / tpeak, 4),
                             "flops": "dense-equivalent 2*M*N*K per matrix"}
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def arith_note(w):
    """What the timed kernels compute in: the JSON line's dtype names the data type in and out."""
    if w.kernel in ("int4_stream_kernel", "nvfp4_stream_kernel", "q8_stream_kernel"):
        return ("bf16 activations in, bf16 out; inside the kernel each run of 64 activations is "
                "held as int16 under one power of two (exact within 2^7 of the run's largest), "
                "integer dot products with the weight codes, fp32 scaling and accumulation")
    if w.kernel in ("bp_stream_kernel", "sa_stream_kernel"):
        return "bf16 in/out; fp32 tables of signed activation sums, fp32 accumulation"
    return "bf16 in/out; bf16 tensor-core operands, fp32 accumulation"


def _src_sha(sources=()):
    """Hash of the CUDA sources a stored counter was taken with (file names under
    bit_weight_gemv_gb300/csrc); the stored value is void once any of them changes."""
    import hashlib
    h = hashlib.sha256()
    for name in sorted(sources):
        p = os.path.join(ROOT, "bit_weight_gemv_gb300", "csrc", name)
        if not os.path.exists(p):
            return None
        with open(p, "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16] if sources else None


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
           "config": {"workload": DEFAULT_WORKLOAD_DESC, "name": "decode_deps", "M": 1,
                      "weight_bytes_per_step": LAYER_BYTES},
           "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": os.cpu_count(),
                            "threads_seen": os_threads(), "kind": "oracle", "sample": sample},
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
    ap.add_argument("--workload", choices=WORKLOADS, default="decode_deps",
                    help="timed step (default: decode through one 4B-class layer, M=1)")
    ap.add_argument("--path", type=int, choices=(0, 1, 2, 3), default=0,
                    help="kernel family: 0 library choice, 1 CUDA cores, 2 tcgen05, 3 warp MMA "
                         "(INT4 and the LM head)")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle timing")
    ap.add_argument("--cpu-child", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_child:  # one CPU-baseline measurement in this process (see cpu_baseline_child)
        # a bounded sample: a pass over 1/64 of every projection's rows sizes the fraction
        # that lets a few passes fit the budget
        _, _, _, t64 = cpu_baseline_oracle(0.0, 1 / 64)
        frac = min(1.0, max(1 / 64, args.cpu_budget / 3 / max(64 * t64, 1e-9)))
        gbs, reps, nbytes, secs = cpu_baseline_oracle(args.cpu_budget, frac)
        print(json.dumps({"gbs": gbs, "reps": reps, "nbytes": nbytes, "secs": secs,
                          "row_fraction": frac, "threads_seen": os_threads()}))
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
