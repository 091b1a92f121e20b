#!/usr/bin/env python3
"""Benchmark of the ConvRot INT8 W8A8 linear on one GB300 (or N, as replicas).

A step is one forward pass of the linear hot path -- online rotation +
per-token INT8 quantization, exact-int32 tcgen05 GEMM, fused dequant to bf16 --
over the single-linear workload at both of its shapes: (M, K, N) =
(2048, 3072, 1024) and (4096, 4096, 4096), group 128, through the C ABI
(ck_int8_linear).  Weights are quantized and laid out once before timing, as a
model load would.  "overlap" repeats the step with overlapped launches across
calls (ck_set_launch_overlap), which the GEMV and MLP measurements use.
Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (oracle/, plain C) on a bounded sample
of the same workload: the only other place this script runs the oracle besides
the cpu_baseline leg.

Secondary objects on the same line (rank 0, after the timed steps): "gemv"
(the M <= 8 decode GEMV sweep), "gemv_lowbit" (the same over the W6A8 / W4A8
weight layouts), "swiglu_mlp" (the fused MLP at both shapes) and
"dit_pass" (45 DiT-shaped blocks of qkv, attention-out, fused MLP and the M = 1
modulation GEMV, every block with its own weights; --no-dit skips it).
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "INT8 ConvRot linear TOPS and % of GB300 dense INT8 peak; M<=8 GEMV HBM GB/s"
UNIT = "TOPS"
WORKLOAD = "convrot_w8a8_linear_2048x3072x1024_and_4096x4096x4096_g128"
N_SETS = 4  # rotating input sets per shape: 4 x ~125 MB > 2 x L2 (129 MB)
NCU_CASES = ("linear_4096", "gemm_4096", "gemm_splitk", "gemm_small", "gemm_k1024", "gateup_4096",
             "quant_4096", "quant_4096_f16",
             "swiglu_4096", "gemv_1", "gemv_2", "gemv_4", "gemv_8", "gemvw6_1", "gemvw6_8",
             "gemvw4_1", "gemvw4_8")


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5000)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-oracle-configs", action="store_true",
                   help="skip the oracle's bounded samples of the MLP, GEMV and DiT workloads")
    p.add_argument("--no-dit", action="store_true",
                   help="skip the DiT-pass measurement (it holds ~8 GB of weights)")
    p.add_argument("--case", default=None,
                   help="profiling mode: run one kernel case a few times and exit (for ncu); "
                        "cases: " + ", ".join(NCU_CASES))
    p.add_argument("--reps", type=int, default=3, help="launches per --case run")
    return p.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(dist, value: float, device) -> float:
    """The largest `value` over all ranks (a MAX all-reduce; `value` itself
    without a process group).  Timings are reported as the slowest rank's."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tops(world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank runs one step's work per step (weak
    scaling), timed by the slowest rank."""
    return world * step_ops() / (ms_per_step * 1e-3) / 1e12


def shapes():
    from swiglu_mlp_group_gb300 import workloads as wl
    return (wl.LINEAR_2048, wl.LINEAR_4096)


def step_ops() -> int:
    return sum(c.ops for c in shapes())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [t.strip() for t in line.split(",")]
            if len(f) >= 9:
                rows.append(f)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------
def oracle_sample(rows_per_shape, seed_offset=0):
    """Times the CPU oracle's linear (rotate, quantize, int64 GEMM, dequant) on
    the first rows of each shape's activations; the oracle's weight
    quantization (load-time work) is outside the timed part.
    Returns (ops, seconds, threads)."""
    import oracle
    from swiglu_mlp_group_gb300 import workloads as wl
    ops, secs = 0, 0.0
    for c, rows in zip(shapes(), rows_per_shape):
        Wq, sw = oracle.quantize_weight(c.W().numpy(), c.g)
        x = wl.bf16_bits(wl.activation(rows, c.K, 1000 * c.seed + 1 + seed_offset,
                                       c.outlier_frac, c.outlier_scale))
        t0 = time.perf_counter()
        oracle.int8_linear(x, Wq, sw, c.g)
        secs += time.perf_counter() - t0
        ops += 2 * rows * c.N * c.K
    return ops, secs, oracle.num_threads()


def oracle_configs_sample(rows=64):
    """The oracle on the host cores over bounded samples of the other workloads:
    the fused MLP at both shapes and one DiT block on the first `rows` token
    rows, the M = 1 decode GEMV whole; the DiT pass is one block's time x 45,
    labelled as an extrapolation.  The oracle's weight quantization (load-time
    work) is outside the timed parts."""
    import numpy as np
    import oracle
    from swiglu_mlp_group_gb300 import workloads as wl

    def timed(fn):
        t0 = time.perf_counter()
        fn()
        return time.perf_counter() - t0

    out = []
    mlp_secs = {}
    for case in (wl.MLP_4096, wl.MLP_2048):
        Wgu_q, sgu = oracle.quantize_weight(
            np.concatenate([case.W_gate().numpy(), case.W_up().numpy()], 0), case.g)
        Wd_q, sd = oracle.quantize_weight(case.W_down().numpy(), case.g)
        x = wl.bf16_bits(case.x()[:rows])
        secs = timed(lambda: oracle.swiglu_mlp(x, Wgu_q, sgu, None, Wd_q, sd, None, case.g))
        mlp_secs[case.name] = secs
        ops = rows * (2 * 2 * case.I * case.H + 2 * case.I * case.H)
        out.append({"workload": case.name, "value": ops / secs / 1e12, "unit": "TOPS",
                    "sample": f"first {rows} of {case.M} token rows", "seconds": secs})
        del Wgu_q, Wd_q
    gv = wl.GEMV_CASES[0]
    Wq, sw = oracle.quantize_weight(gv.W().numpy(), gv.g)
    x = wl.bf16_bits(gv.x())
    secs = timed(lambda: oracle.int8_linear(x, Wq, sw, gv.g))
    out.append({"workload": gv.name, "value": gv.algorithmic_bytes() / secs / 1e9, "unit": "GB/s",
                "sample": "the whole call", "seconds": secs})
    blk = wl.DIT_BLOCK
    block_secs = mlp_secs[wl.MLP_4096.name]  # the block's MLP is the 4096 x 3072 x 12288 one
    block_ops = rows * (2 * 2 * blk.mlp * blk.hidden + 2 * blk.mlp * blk.hidden)
    xb = wl.bf16_bits(wl.activation(rows, blk.hidden, 4243))
    for i, (_, k, n) in enumerate(blk.linears):
        Wq, sw = oracle.quantize_weight(wl.weight(n, k, 4300 + i).numpy(), blk.g)
        block_secs += timed(lambda: oracle.int8_linear(xb, Wq, sw, blk.g))
        block_ops += 2 * rows * k * n
    mk, mn = blk.modulation
    Wq, sw = oracle.quantize_weight(wl.weight(mn, mk, 4310).numpy(), blk.g)
    xm = wl.bf16_bits(wl.activation(1, mk, 4244))
    block_secs += timed(lambda: oracle.int8_linear(xm, Wq, sw, blk.g))
    block_ops += 2 * mk * mn
    out.append({"workload": f"dit_pass_{blk.blocks}_blocks_M{blk.M}_H{blk.hidden}_I{blk.mlp}_g{blk.g}",
                "value": block_ops / block_secs / 1e12, "unit": "TOPS",
                "sample": f"one block on the first {rows} of {blk.M} token rows (and the M = 1 "
                          f"modulation); the pass extrapolated as {blk.blocks} x that block",
                "seconds": block_secs,
                "pass_seconds_extrapolated": blk.blocks * block_secs * blk.M / rows})
    return out, oracle.num_threads()


def run_reference(args, world, rank):
    if rank != 0:
        return
    rows = (256, 128)  # bounded sample per step (about a second of CPU work)
    for i in range(args.warmup):
        oracle_sample(rows, i)
    ops = secs = 0.0
    threads = 1
    for i in range(args.steps):
        o, s, threads = oracle_sample(rows, 100 + i)
        ops += o
        secs += s
    value = ops / secs / 1e12
    sample = f"{rows[0]} rows of 2048x3072->1024 + {rows[1]} rows of 4096x4096->4096 per step"
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def _code_only(text):
    """C++ source without comments or blank lines: what the kernels are compiled from."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*", "", line).rstrip() for line in text.splitlines())
    return "\n".join(line for line in lines if line)


def gemm_traffic_from_profile():
    """DRAM bytes per launch of the GEMM kernel from the committed ncu summary,
    if it was taken on the kernel source as it is now (else None)."""
    path = os.path.join(ROOT, "profiles", "gemm_tcgen05_linear_4096_traffic.txt")
    csrc = os.path.join(ROOT, "swiglu_mlp_group_gb300", "csrc")
    srcs = [os.path.join(csrc, f) for f in ("gemm_tcgen05.cu", "gemm_tcgen05_2sm.cu",
                                             "gemm_issue.cuh", "gemm_epilogue.cuh", "ptx.cuh")]
    if not os.path.exists(path):
        return None
    kv = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    digest = hashlib.sha256(b"".join(_code_only(open(f).read()).encode() for f in srcs)).hexdigest()[:16]
    if kv.get("kernel_source_sha256_16") != digest:
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d.get("bf16_tflops"), d.get("hbm_gbs"), "measured"
    return 1900.0, 6800.0, "fallback"


def graph_us(torch, cap, fn, overlap, ck, reps=40):
    """Median time per call (us) of `reps` back-to-back fn(j) calls captured in
    one CUDA graph on stream `cap`, launched with ck_set_launch_overlap(overlap)."""
    ck.set_launch_overlap(overlap)
    try:
        with torch.cuda.stream(cap):
            for j in range(3):
                fn(j)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=cap):
            for j in range(reps):
                fn(j)
    finally:
        ck.set_launch_overlap(False)
    gr.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ts = []
    for _ in range(5):
        e0.record()
        gr.replay()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) / reps)
    return statistics.median(ts) * 1e3


def bench_gemv(ck, torch, dev, cap, peak_hbm, bits=8, Ms=(1, 2, 4, 8)):
    """Small-M decode GEMV sweep over the three weight shapes, each a whole
    small-M GEMV call (activation quantizer + GEMV, or one kernel where the
    CTAs quantize x themselves), 4 rotating packed weights per shape (> 2 x L2),
    CUDA-graph replay.  bits: the weight code width (8: INT8; 6 / 4: the W6A8 /
    W4A8 layouts)."""
    from swiglu_mlp_group_gb300 import workloads as wl
    layout = ck.GEMV_LAYOUT_OF_BITS[bits]
    out = []
    shapes_nk = [(12288, 4096), (4096, 12288), (18432, 3072)]
    for (N, K) in shapes_nk:
        packs = []
        for i in range(N_SETS):
            Wq, sw = ck.quantize_weight_bits(wl.weight(N, K, 900 + 7 * i + K).to(dev), 128, bits)
            packs.append(ck.prepare_weight(Wq, sw, layout))
            del Wq, sw
        wbytes = N * K * bits // 8 + 4 * N
        for M in Ms:
            x = wl.activation(M, K, 950 + M).to(dev)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ws = torch.empty(ck.workspace_bytes(ck.CK_OP_GEMV_SMALLM, M, K, N), dtype=torch.uint8,
                             device=dev)
            xq8, sx = ck.rotate_quantize_act(x, 128)
            torch.cuda.synchronize()
            call = lambda j: ck.gemv_smallM(x, packs[j % N_SETS], N, 128, out=y, workspace=ws,
                                            stream=cap, wlayout=layout)
            kern = lambda j: ck.packed_gemv_dequant(xq8, sx, packs[j % N_SETS], layout, N, out=y,
                                                    stream=cap)
            nbytes = wbytes + 2 * M * K + 2 * M * N
            kbytes = wbytes + M * K + 4 * M + 2 * M * N  # int8 codes in
            t = {ov: (graph_us(torch, cap, call, ov, ck), graph_us(torch, cap, kern, ov, ck))
                 for ov in (False, True)}
            us, kus = t[True]
            # one kernel where every CTA quantizes x itself (the rule in include/ck.h,
            # overlapped launches): M = 1 with K <= 16384, M = 2 with K <= 8192
            fused = (M == 1 and K <= 16384) or (M == 2 and K <= 8192)
            out.append({"M": M, "N": N, "K": K, "us": us, "GB/s": nbytes / (us * 1e-6) / 1e9,
                        "frac": nbytes / (us * 1e-6) / 1e9 / peak_hbm,
                        "launches_per_call": 1 if fused else 2, "kernel_us": kus,
                        "kernel_GB/s": kbytes / (kus * 1e-6) / 1e9,
                        "kernel_frac": kbytes / (kus * 1e-6) / 1e9 / peak_hbm,
                        "no_overlap": {"us": t[False][0], "kernel_us": t[False][1],
                                       "frac": nbytes / (t[False][0] * 1e-6) / 1e9 / peak_hbm,
                                       "kernel_frac": kbytes / (t[False][1] * 1e-6) / 1e9 / peak_hbm}})
        del packs
        torch.cuda.empty_cache()
    wdesc = "N*K" if bits == 8 else f"N*K*{bits}/8"
    return {"unit": "GB/s", "peak": peak_hbm, "peak_source": "measured HBM copy",
            "weight_bits": bits,
            "bytes": f"{wdesc} + 4N packed weight + 2MK x + 2MN y per call",
            "how": "40 back-to-back calls per CUDA graph, 4 rotating packed weights; headline "
                   "numbers with ck_set_launch_overlap(1) (weights settled, each call overlaps "
                   "the tail of the one ahead), 'no_overlap' with it off",
            "cases": out}


def gemm_alone_ms(ck, torch, cap, items, reps=20):
    """Median per-launch ms of int8_gemm_dequant alone over `items` (tuples of
    codes16, sx, W16, sw, out), rotated per launch, replayed in a CUDA graph."""
    with torch.cuda.stream(cap):
        for j in range(3):
            a, sx, w, sw, out = items[j % len(items)]
            ck.int8_gemm_dequant(a, sx, w, sw, out=out, stream=cap)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        for j in range(reps):
            a, sx, w, sw, out = items[j % len(items)]
            ck.int8_gemm_dequant(a, sx, w, sw, out=out, stream=cap)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ts = []
    for _ in range(5):
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) / reps)
    return statistics.median(ts)


def gemm_entry(M, N, K, ms, peak_tf):
    tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
    return {"M": M, "N": N, "K": K, "us": ms * 1e3, "TFLOP/s": tf, "frac": tf / peak_tf}


def bench_mlp(ck, torch, dev, cap):
    """The fused SwiGLU MLP (packed gate|up linear, swiglu-quantized down
    linear) at both workload shapes, 2 rotating weight sets (> 2 x L2), CUDA
    graph replay of ck_swiglu_mlp; "glu": the same with the SwiGLU product
    formed in the gate|up GEMM's epilogue (CK_WLAYOUT_GEMM_F16_GLU)."""
    from swiglu_mlp_group_gb300 import workloads as wl
    out = []
    for case in (wl.MLP_4096, wl.MLP_2048):
        sets = []
        for i in range(2):
            Wgu = torch.cat([wl.weight(case.I, case.H, 1000 * case.seed + 2 + 31 * i),
                             wl.weight(case.I, case.H, 1000 * case.seed + 3 + 31 * i)], 0)
            Wgu_q, sgu = ck.quantize_weight(Wgu.to(dev), case.g)
            del Wgu
            Wd_q, sd = ck.quantize_weight(wl.weight(case.H, case.I, 1000 * case.seed + 4 + 31 * i)
                                          .to(dev), case.g)
            sets.append({ck.CK_WLAYOUT_GEMM_F16: ck.prepare_weight(Wgu_q, sgu, ck.CK_WLAYOUT_GEMM_F16),
                         ck.CK_WLAYOUT_GEMM_F16_GLU: ck.prepare_weight(Wgu_q, sgu,
                                                                       ck.CK_WLAYOUT_GEMM_F16_GLU),
                         "sgu": sgu, "Wd": ck.prepare_weight(Wd_q, sd, ck.CK_WLAYOUT_GEMM_F16),
                         "sd": sd})
            del Wgu_q, Wd_q
        x = case.x().to(dev)
        y = torch.empty((case.M, case.H), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(ck.workspace_bytes(ck.CK_OP_SWIGLU_MLP, case.M, case.H, case.I,
                                            ck.CK_WLAYOUT_GEMM_F16), dtype=torch.uint8, device=dev)
        reps = 6

        def timed_ms(layout):
            def call(j, stream):
                st = sets[j % 2]
                ck.swiglu_mlp(x, st[layout], st["sgu"], st["Wd"], st["sd"], case.g, wlayout=layout,
                              out=y, workspace=ws, stream=stream)

            torch.cuda.synchronize()
            ck.set_launch_overlap(True)  # the weights are settled
            try:
                with torch.cuda.stream(cap):
                    for j in range(2):
                        call(j, cap)
                torch.cuda.synchronize()
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr, stream=cap):
                    for j in range(reps):
                        call(j, cap)
            finally:
                ck.set_launch_overlap(False)
            gr.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ts = []
            for _ in range(5):
                e0.record()
                gr.replay()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1) / reps)
            return statistics.median(ts)

        ms = timed_ms(ck.CK_WLAYOUT_GEMM_F16)
        ms_glu = timed_ms(ck.CK_WLAYOUT_GEMM_F16_GLU)
        # the two GEMMs alone, on codes quantized outside the timed part (x for the
        # gate|up GEMM, a stand-in silu(gate) * up for the down GEMM)
        peak_tf = measured_peaks()[0]
        xq16, sx = ck.rotate_quantize_act_f16(x, case.g)
        aq16, sa = ck.rotate_quantize_act_f16(wl.activation(case.M, case.I, 1000 * case.seed + 9).to(dev), case.g)
        h = torch.empty((case.M, 2 * case.I), dtype=torch.bfloat16, device=dev)
        gu = gemm_alone_ms(ck, torch, cap, [(xq16, sx, st[ck.CK_WLAYOUT_GEMM_F16], st["sgu"], h) for st in sets])
        dn = gemm_alone_ms(ck, torch, cap, [(aq16, sa, st["Wd"], st["sd"], y) for st in sets])
        del h
        out.append({"workload": case.name, "M": case.M, "H": case.H, "I": case.I, "ms": ms,
                    "TOPS": case.ops / (ms * 1e-3) / 1e12, "launches_per_call": 4,
                    "glu": {"ms": ms_glu, "TOPS": case.ops / (ms_glu * 1e-3) / 1e12,
                            "launches_per_call": 4},
                    "gemm_gateup": gemm_entry(case.M, 2 * case.I, case.H, gu, peak_tf),
                    "gemm_down": gemm_entry(case.M, case.H, case.I, dn, peak_tf)})
        del sets, ws
        torch.cuda.empty_cache()
    return out


def bench_dit_pass(ck, torch, dev, cap):
    """One DiT-shaped forward pass: 45 blocks of {qkv 3072 -> 9216, attention-out
    3072 -> 3072, the fused SwiGLU MLP 3072 -> 2 x 12288 -> 3072} at M = 4096
    plus the modulation linear 3072 -> 18432 at M = 1 (small-M GEMV), every
    block with its own weights (~16 GB resident); one bf16 input per distinct
    K, reused across layers (the shapes do not chain); one stream, CUDA graph."""
    from swiglu_mlp_group_gb300 import workloads as wl
    blk = wl.DIT_BLOCK
    M, H, I, g = blk.M, blk.hidden, blk.mlp, blk.g
    gen = torch.Generator(device=dev)
    gen.manual_seed(4242)

    def qweight(N, K, layout):
        W = torch.randn(N, K, device=dev, generator=gen) * (1.0 / math.sqrt(K))
        Wq, sw = ck.quantize_weight(W, g)
        del W
        return ck.prepare_weight(Wq, sw, layout), sw

    F16, PACK = ck.CK_WLAYOUT_GEMM_F16, ck.CK_WLAYOUT_GEMV_PACKED
    (_, _, qkv_n), (_, _, ao_n) = blk.linears
    mod_k, mod_n = blk.modulation
    blocks = []
    for _ in range(blk.blocks):
        blocks.append({"qkv": qweight(qkv_n, H, F16), "ao": qweight(ao_n, H, F16),
                       "gu": qweight(2 * I, H, F16), "dn": qweight(H, I, F16),
                       "mod": qweight(mod_n, mod_k, PACK)})
    weight_bytes = sum(t.numel() * t.element_size() for b in blocks for (w, s) in b.values()
                       for t in (w, s))
    x = wl.activation(M, H, 4243).to(dev)
    xm = wl.activation(1, mod_k, 4244).to(dev)
    y_qkv = torch.empty((M, qkv_n), dtype=torch.bfloat16, device=dev)
    y_ao = torch.empty((M, ao_n), dtype=torch.bfloat16, device=dev)
    y_mlp = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    y_mod = torch.empty((1, mod_n), dtype=torch.bfloat16, device=dev)
    ws_lin = torch.empty(max(ck.workspace_bytes(ck.CK_OP_INT8_LINEAR, M, H, qkv_n, F16),
                             ck.workspace_bytes(ck.CK_OP_INT8_LINEAR, M, H, ao_n, F16)),
                         dtype=torch.uint8, device=dev)
    ws_mlp = torch.empty(ck.workspace_bytes(ck.CK_OP_SWIGLU_MLP, M, H, I, F16), dtype=torch.uint8,
                         device=dev)
    ws_mod = torch.empty(ck.workspace_bytes(ck.CK_OP_GEMV_SMALLM, 1, mod_k, mod_n),
                         dtype=torch.uint8, device=dev)
    parts = {
        "qkv": lambda b, s: ck.int8_linear(x, b["qkv"][0], b["qkv"][1], g, wlayout=F16, out=y_qkv,
                                           workspace=ws_lin, stream=s),
        "attn_out": lambda b, s: ck.int8_linear(x, b["ao"][0], b["ao"][1], g, wlayout=F16,
                                                out=y_ao, workspace=ws_lin, stream=s),
        "swiglu_mlp": lambda b, s: ck.swiglu_mlp(x, b["gu"][0], b["gu"][1], b["dn"][0],
                                                 b["dn"][1], g, wlayout=F16, out=y_mlp,
                                                 workspace=ws_mlp, stream=s),
        "modulation_gemv": lambda b, s: ck.gemv_smallM(xm, b["mod"][0], mod_n, g, out=y_mod,
                                                       workspace=ws_mod, stream=s),
    }
    ops = {"qkv": 2 * M * H * qkv_n, "attn_out": 2 * M * H * ao_n,
           "swiglu_mlp": 2 * M * H * 2 * I + 2 * M * I * H, "modulation_gemv": 2 * mod_k * mod_n}

    torch.cuda.synchronize()  # every block's weights settled

    def graph_ms(calls):
        ck.set_launch_overlap(True)
        try:
            with torch.cuda.stream(cap):
                for b in blocks[:2]:
                    for c in calls:
                        c(b, cap)
            torch.cuda.synchronize()
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=cap):
                for b in blocks:
                    for c in calls:
                        c(b, cap)
        finally:
            ck.set_launch_overlap(False)
        gr.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ts = []
        for _ in range(3):
            e0.record()
            gr.replay()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        del gr
        return statistics.median(ts)

    pass_ms = graph_ms(list(parts.values()))
    per_part = {k: graph_ms([fn]) for k, fn in parts.items()}
    total_ops = blk.blocks * sum(ops.values())
    out = {"workload": f"dit_pass_{blk.blocks}_blocks_M{M}_H{H}_I{I}_g{g}", "ms": pass_ms,
           "TOPS": total_ops / (pass_ms * 1e-3) / 1e12, "ops": total_ops,
           "weights_GB_resident": weight_bytes / 1e9, "calls_per_block": 4,
           "parts_ms": per_part,
           "parts_TOPS": {k: blk.blocks * ops[k] / (per_part[k] * 1e-3) / 1e12 for k in parts}}
    del blocks
    torch.cuda.empty_cache()
    return out


def run_case(args):
    """Small, self-contained runs of single kernels for Nsight Compute captures:
    each case builds its inputs (seeded, synthetic), runs its kernels --reps
    times and exits; device memory stays within a few GB, so a capture of one
    launch ends by itself.
      linear_4096     ConvRot linear at M = K = N = 4096 (quantize + GEMM)
      gemm_4096       the GEMM alone on pre-quantized codes, M = K = N = 4096
      gemm_splitk     the same at M = 2048, N = 1024, K = 12288 (K split between two CTA pairs)
      gemm_small      the same at M = 2048, N = 1024, K = 3072 (the linear step's small GEMM)
      gemm_k1024      the same at M = 2048, N = 3072, K = 1024 (the 2048-token MLP's down GEMM)
      gateup_4096     the packed gate|up linear of the MLP, M=4096, K=3072, N=24576
      quant_4096      the activation quantizer alone, M = K = 4096 (INT8 codes)
      quant_4096_f16  the same writing the GEMM's fp16-held codes
      swiglu_4096     the swiglu activation quantizer, M=4096, I=12288 (fp16-held codes)
      gemv_<M>        small-M GEMV call over the packed layout, N=12288, K=4096
      gemvw<b>_<M>    the same over the W6A8 / W4A8 layout (b = 6, 4)"""
    import torch
    import swiglu_mlp_group_gb300 as ck
    from swiglu_mlp_group_gb300 import workloads as wl
    if args.case not in NCU_CASES:
        raise SystemExit(f"unknown case {args.case}; cases: {', '.join(NCU_CASES)}")
    ck.build()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    g, a = 128, args.case
    if a in ("linear_4096", "gemm_4096", "gemm_splitk", "gemm_small", "gemm_k1024", "gateup_4096"):
        M, K, N = {"gateup_4096": (4096, 3072, 24576), "gemm_splitk": (2048, 12288, 1024),
                   "gemm_small": (2048, 3072, 1024), "gemm_k1024": (2048, 1024, 3072)}.get(
            a, (4096, 4096, 4096))
        x = wl.activation(M, K, 11, 0.005, 30.0).to(dev)
        Wq, sw = ck.quantize_weight(wl.weight(N, K, 12).to(dev), g)
        W16 = ck.prepare_weight(Wq, sw, ck.CK_WLAYOUT_GEMM_F16)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        if a in ("gemm_4096", "gemm_splitk", "gemm_small", "gemm_k1024"):
            xq16, sx = ck.rotate_quantize_act_f16(x, g)
            for _ in range(args.reps):
                ck.int8_gemm_dequant(xq16, sx, W16, sw, out=y)
        else:
            for _ in range(args.reps):
                ck.int8_linear(x, W16, sw, g, wlayout=ck.CK_WLAYOUT_GEMM_F16, out=y)
    elif a in ("quant_4096", "quant_4096_f16"):
        x = wl.activation(4096, 4096, 13, 0.005, 30.0).to(dev)
        quant = ck.rotate_quantize_act if a == "quant_4096" else ck.rotate_quantize_act_f16
        for _ in range(args.reps):
            quant(x, g)
    elif a == "swiglu_4096":
        h = wl.activation(4096, 2 * 12288, 14).to(dev)
        for _ in range(args.reps):
            ck.rotate_quantize_act_f16(h, g, act="swiglu")
    else:
        head, m = a.split("_")
        M, bits = int(m), (8 if head == "gemv" else int(head[len("gemvw"):]))
        layout = ck.GEMV_LAYOUT_OF_BITS[bits]
        N, K = 12288, 4096
        x = wl.activation(M, K, 15).to(dev)
        Wq, sw = ck.quantize_weight_bits(wl.weight(N, K, 16).to(dev), g, bits)
        Wp = ck.prepare_weight(Wq, sw, layout)
        for _ in range(args.reps):
            ck.gemv_smallM(x, Wp, N, g, wlayout=layout)
    torch.cuda.synchronize()
    if ck.poll_device_status() != ck.CK_OK:
        raise SystemExit("a device-side wait timed out")


def bench_quantize(ck, torch, dev, cap, peak_hbm):
    """The activation quantizer alone (ck_rotate_quantize_act, INT8 codes out)
    on the linear workload's two activations and the MLP's swiglu input, 4
    rotating inputs per shape (> L2 for the 4096-row ones), 40 back-to-back
    launches per CUDA graph.  Algorithmic bytes: 2MK read + MK codes + 4M
    scales (act none); 4MI read + MI codes + 4M scales (swiglu)."""
    from swiglu_mlp_group_gb300 import workloads as wl
    out = []
    for (M, K, act) in ((4096, 4096, "none"), (2048, 3072, "none"), (4096, 12288, "swiglu")):
        cols = 2 * K if act == "swiglu" else K
        xs = [wl.activation(M, cols, 960 + i, 0.005, 30.0).to(dev) for i in range(N_SETS)]
        xq = torch.empty((M, K), dtype=torch.int8, device=dev)
        sx = torch.empty((M,), dtype=torch.float32, device=dev)
        actc = ck.CK_ACT_SWIGLU if act == "swiglu" else ck.CK_ACT_NONE

        def call(j):
            ck._check(ck.ck_rotate_quantize_act(xs[j % N_SETS].data_ptr(), M, K, cols, actc, 128,
                                                xq.data_ptr(), sx.data_ptr(), cap.cuda_stream),
                      "ck_rotate_quantize_act")

        us = graph_us(torch, cap, call, False, ck)
        us_ov = graph_us(torch, cap, call, True, ck)
        nbytes = (4 if act == "swiglu" else 2) * M * K + M * K + 4 * M
        out.append({"M": M, "K": K, "act": act, "us": us, "GB/s": nbytes / (us * 1e-6) / 1e9,
                    "frac": nbytes / (us * 1e-6) / 1e9 / peak_hbm, "bytes": nbytes,
                    "overlapped": {"us": us_ov, "frac": nbytes / (us_ov * 1e-6) / 1e9 / peak_hbm}})
        del xs
    return {"unit": "GB/s", "peak": peak_hbm, "peak_source": "measured HBM copy",
            "bytes": "algorithmic: input read once, INT8 codes and f32 scales written",
            "how": ("40 back-to-back launches per CUDA graph, 4 rotating inputs; 'overlapped': the "
                    "same with programmatic dependent launches (each launch still waits for the one "
                    "before it to finish before reading its input)"), "cases": out}


ENQUEUE_C = r"""
#include <stdio.h>
#include <stdint.h>
#include <time.h>
#include <cuda_runtime.h>
#include "ck.h"
static double now_us(void) {
    struct timespec t; clock_gettime(CLOCK_MONOTONIC, &t);
    return t.tv_sec * 1e6 + t.tv_nsec * 1e-3;
}
int main(void) {
    cudaStream_t s; cudaStreamCreate(&s);
    void *x, *w, *sw, *y, *ws, *wp;
    const int64_t M = 2048, K = 3072, N = 1024, GN = 12288, GK = 4096;
    cudaMalloc(&x, M * K * 2); cudaMalloc(&w, N * K); cudaMalloc(&sw, GN * 4);
    cudaMalloc(&y, M * N * 2); cudaMalloc(&ws, 64 << 20);
    size_t pb = ck_prepared_weight_bytes(CK_WLAYOUT_GEMV_PACKED, GN, GK);
    cudaMalloc(&wp, pb);
    cudaMemset(x, 0, M * K * 2); cudaMemset(w, 0, N * K); cudaMemset(sw, 0, GN * 4);
    cudaMemset(wp, 0, pb);
    const int reps = 200;
    double t_lin = 0, t_gemv = 0;
    for (int pass = 0; pass < 2; ++pass) {
        cudaStreamSynchronize(s);
        double t0 = now_us();
        for (int i = 0; i < reps; ++i)
            if (ck_int8_linear(x, M, K, K, CK_ACT_NONE, w, CK_WLAYOUT_ROWMAJOR_I8, (const float *)sw,
                               N, 128, NULL, NULL, y, ws, 64 << 20, (ck_stream_t)s) != CK_OK) return 2;
        t_lin = (now_us() - t0) / reps;
        cudaStreamSynchronize(s);
        t0 = now_us();
        for (int i = 0; i < reps; ++i)
            if (ck_int8_gemv_smallM(x, 1, GK, GK, CK_ACT_NONE, wp, GN, 128, NULL, NULL, y, ws,
                                    64 << 20, (ck_stream_t)s) != CK_OK) return 3;
        t_gemv = (now_us() - t0) / reps;
    }
    cudaStreamSynchronize(s);
    if (ck_poll_device_status((ck_stream_t)s) != CK_OK) return 4;
    printf("%.4f %.4f\n", t_lin, t_gemv);
    return 0;
}
"""


def enqueue_cost(ck):
    """Host microseconds per call, measured in C (no Python in the loop): 200
    ck_int8_linear calls (2048 x 3072 -> 1024, two kernels each) and 200
    ck_int8_gemv_smallM calls (M = 1, 12288 x 4096, one kernel), each loop
    timed with CLOCK_MONOTONIC around the enqueues only (the GPU runs behind)."""
    import shutil
    cc = shutil.which("gcc") or shutil.which("cc")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    if cc is None:
        return None
    d = tempfile.mkdtemp()
    src, exe = os.path.join(d, "enqueue.c"), os.path.join(d, "enqueue")
    with open(src, "w") as f:
        f.write(ENQUEUE_C)
    libdir = os.path.dirname(ck.library_path())
    r = subprocess.run([cc, "-O2", src, "-o", exe, "-I", os.path.join(ROOT, "include"),
                        "-I", os.path.join(cuda, "include"), "-L", os.path.join(cuda, "lib64"),
                        "-L", libdir, "-lck_gb300", "-lcudart", f"-Wl,-rpath,{libdir}",
                        f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"],
                       capture_output=True, text=True)
    if r.returncode != 0:
        return {"error": r.stderr.strip()[-300:]}
    r = subprocess.run([exe], capture_output=True, text=True,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES=os.environ.get(
                           "CUDA_VISIBLE_DEVICES", "0")))
    shutil.rmtree(d, ignore_errors=True)
    if r.returncode != 0:
        return {"error": f"harness exited {r.returncode}"}
    lin, gemv = (float(v) for v in r.stdout.split())
    return {"ck_int8_linear_us": lin, "ck_int8_gemv_smallM_us": gemv,
            "how": "C harness (gcc, libck_gb300.so, cudart): 200 calls per loop, host "
                   "CLOCK_MONOTONIC around the enqueues; linear 2048x3072->1024 on the INT8 "
                   "weight, GEMV M = 1 over 12288x4096 packed"}


def run_ours(args, world, rank, local):
    import torch
    import swiglu_mlp_group_gb300 as ck

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    ck.build()
    if ck.ck_device_check() != ck.CK_OK:
        raise SystemExit("bench.py: the device is not a compute capability 10.3 GB300")
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    cases = shapes()
    stream = torch.cuda.current_stream()
    sets = []  # per set: list over shapes of dict of device tensors
    for i in range(N_SETS):
        per = []
        for c in cases:
            x = c.x() if i == 0 else None
            if x is None:
                from swiglu_mlp_group_gb300 import workloads as wl
                x = wl.activation(c.M, c.K, 1000 * c.seed + 1 + 17 * i, c.outlier_frac,
                                  c.outlier_scale)
            from swiglu_mlp_group_gb300 import workloads as wl
            W = c.W() if i == 0 else wl.weight(c.N, c.K, 1000 * c.seed + 2 + 17 * i)
            Wq, sw = ck.quantize_weight(W.to(dev), c.g)
            W16 = ck.prepare_weight(Wq, sw, ck.CK_WLAYOUT_GEMM_F16)
            del Wq
            ws = torch.empty(ck.workspace_bytes(ck.CK_OP_INT8_LINEAR, c.M, c.K, c.N,
                                                ck.CK_WLAYOUT_GEMM_F16), dtype=torch.uint8,
                             device=dev)
            per.append({"case": c, "x": x.to(dev), "W16": W16, "sw": sw, "ws": ws,
                        "y": torch.empty((c.M, c.N), dtype=torch.bfloat16, device=dev),
                        "x_host": x.pin_memory() if i == 0 else None})
        sets.append(per)
    torch.cuda.synchronize()

    def step(per, s):
        for d in per:
            c = d["case"]
            ck._check(ck.ck_int8_linear(d["x"].data_ptr(), c.M, c.K, c.K, ck.CK_ACT_NONE,
                                        d["W16"].data_ptr(), ck.CK_WLAYOUT_GEMM_F16,
                                        d["sw"].data_ptr(), c.N, c.g, None, None,
                                        d["y"].data_ptr(), d["ws"].data_ptr(), d["ws"].numel(),
                                        s.cuda_stream),
                      "ck_int8_linear")

    # one CUDA graph per input set: a step replays one graph (4 kernels).  The
    # headline graphs use the default launches (each call's GEMM already starts
    # under its quantizer's tail); a second set captured with overlapped
    # launches across calls (the weights were prepared and synchronized above)
    # is timed for reference: it does not help this step's long kernels.
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)

    def capture_steps(overlap):
        ck.set_launch_overlap(overlap)
        try:
            with torch.cuda.stream(cap):
                for per in sets:
                    step(per, cap)
            torch.cuda.synchronize()
            out = []
            for per in sets:
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr, stream=cap):
                    step(per, cap)
                out.append(gr)
        finally:
            ck.set_launch_overlap(False)
        return out

    graphs_overlap = capture_steps(True)
    graphs = capture_steps(False)
    stream.wait_stream(cap)
    launches_per_step = 2 * len(cases)

    for gs in (graphs_overlap, graphs):
        for i in range(args.warmup):
            gs[i % N_SETS].replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        graphs_overlap[i % N_SETS].replay()
    e1.record()
    torch.cuda.synchronize()
    overlap_ms = e0.elapsed_time(e1) / args.steps
    del graphs_overlap

    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0.record()
    for i in range(args.steps):
        graphs[i % N_SETS].replay()
    e1.record()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    elapsed_ms = max_over_ranks(dist, e0.elapsed_time(e1), dev)
    clock_info = clocks.stop() if clocks else None
    if ck.poll_device_status() != ck.CK_OK:
        raise SystemExit("bench.py: a device-side wait timed out; results invalid")
    ms_per_step = elapsed_ms / args.steps
    value = whole_job_tops(world, ms_per_step)

    # ---- dominant kernel (the 4096^3 GEMM) timed alone, live, same stream
    big = [per[1] for per in sets]
    c = big[0]["case"]
    codes = []
    for d in big:
        xq16, sx = ck.rotate_quantize_act_f16(d["x"], c.g)
        codes.append((xq16, sx))
    reps = 20
    with torch.cuda.stream(cap):
        for j in range(3):
            d, (xq16, sx) = big[j % N_SETS], codes[j % N_SETS]
            ck.int8_gemm_dequant(xq16, sx, d["W16"], d["sw"], out=d["y"], stream=cap)
    torch.cuda.synchronize()
    g_gemm = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_gemm, stream=cap):
        for j in range(reps):
            d, (xq16, sx) = big[j % N_SETS], codes[j % N_SETS]
            ck.int8_gemm_dequant(xq16, sx, d["W16"], d["sw"], out=d["y"], stream=cap)
    g_gemm.replay()
    torch.cuda.synchronize()
    gt = []
    for _ in range(5):
        e0.record()
        g_gemm.replay()
        e1.record()
        torch.cuda.synchronize()
        gt.append(e0.elapsed_time(e1) / reps)
    gemm_ms = statistics.median(gt)
    peak_tf, peak_hbm, peak_src = measured_peaks()
    achieved_tf = 2.0 * c.M * c.N * c.K / (gemm_ms * 1e-3) / 1e12
    traffic = gemm_traffic_from_profile()
    roofline = {"bound": "tensor", "kernel": "gemm_codes_pair_kernel (tcgen05 kind::f16 cta_group::2, 4096^3)",
                "achieved": achieved_tf, "peak": peak_tf, "unit": "TFLOP/s",
                "frac": achieved_tf / peak_tf, "peak_source": f"{peak_src} bf16 dense (burst)",
                "traffic": traffic, "launch_ms": gemm_ms}
    # the step's other GEMM (2048 x 3072 -> 1024) alone, the same way
    small = [per[0] for per in sets]
    cs = small[0]["case"]
    small_items = []
    for d in small:
        xq16, sx = ck.rotate_quantize_act_f16(d["x"], cs.g)
        small_items.append((xq16, sx, d["W16"], d["sw"], d["y"]))
    gemm_small = gemm_entry(cs.M, cs.N, cs.K, gemm_alone_ms(ck, torch, cap, small_items), peak_tf)
    gemm_small["bf16_burst_peak"] = peak_tf
    int8_peak = ck.measure_int8_mma_tops()
    engine_peak = ck.measure_tcgen05_f16_tflops()
    gemv = bench_gemv(ck, torch, dev, cap, peak_hbm) if rank == 0 else None
    gemv_lowbit = ({f"w{b}a8": bench_gemv(ck, torch, dev, cap, peak_hbm, bits=b, Ms=(1, 2, 8))
                    for b in (6, 4)} if rank == 0 else None)
    quantize = bench_quantize(ck, torch, dev, cap, peak_hbm) if rank == 0 else None
    enqueue = enqueue_cost(ck) if rank == 0 else None
    mlp = bench_mlp(ck, torch, dev, cap) if rank == 0 else None
    dit = bench_dit_pass(ck, torch, dev, cap) if rank == 0 and not args.no_dit else None

    # ---- end to end through the C ABI with host buffers: every step copies its
    # inputs from pinned host memory and its outputs back; one step's copies
    # overlap the compute and the copies of its neighbours (NB buffers, three
    # streams), as a serving loop would run it.  The C entry point is called
    # directly with cached pointers so that the host keeps ahead of the GPU.
    NB = 3
    d2 = list(sets[0])
    x_host = [d["x_host"] for d in d2]
    y_host = [[torch.empty(d["y"].shape, dtype=torch.bfloat16).pin_memory() for d in d2]
              for _ in range(NB)]
    x_dev = [[torch.empty_like(d["x"]) for d in d2] for _ in range(NB)]
    y_dev = [[torch.empty_like(d["y"]) for d in d2] for _ in range(NB)]
    h2d = sum(x.numel() * 2 for x in x_host)
    d2h = sum(y.numel() * 2 for y in y_host[0])
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(NB)]
    ev_cmp = [torch.cuda.Event() for _ in range(NB)]
    ev_out = [torch.cuda.Event() for _ in range(NB)]
    linear_args = [[(xd.data_ptr(), d["case"].M, d["case"].K, d["case"].K, ck.CK_ACT_NONE,
                     d["W16"].data_ptr(), ck.CK_WLAYOUT_GEMM_F16, d["sw"].data_ptr(), d["case"].N,
                     d["case"].g, None, None, yd.data_ptr(), d["ws"].data_ptr(), d["ws"].numel(),
                     s_cmp.cuda_stream)
                    for d, xd, yd in zip(d2, x_dev[b], y_dev[b])] for b in range(NB)]
    c_linear = ck.ck_int8_linear

    def e2e_step(i, compute=True):
        b = i % NB
        if i >= NB:
            s_in.wait_event(ev_cmp[b])      # x_dev[b] consumed by step i - NB
        with torch.cuda.stream(s_in):
            for xd, xh in zip(x_dev[b], x_host):
                xd.copy_(xh, non_blocking=True)
        ev_in[b].record(s_in)
        s_cmp.wait_event(ev_in[b])
        if i >= NB:
            s_cmp.wait_event(ev_out[b])     # y_dev[b] read back by step i - NB
        for a in (linear_args[b] if compute else ()):
            st = c_linear(*a)
            if st != ck.CK_OK:
                raise SystemExit(f"bench.py: ck_int8_linear returned {ck.status_string(st)}")
        ev_cmp[b].record(s_cmp)
        s_out.wait_event(ev_cmp[b])
        with torch.cuda.stream(s_out):
            for yh, yd in zip(y_host[b], y_dev[b]):
                yh.copy_(yd, non_blocking=True)
        ev_out[b].record(s_out)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    for i in range(args.steps):
        e2e_step(i)
    t_enq = time.perf_counter()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(dist, (time.perf_counter() - t0) * 1e3 / args.steps, dev)
    enqueue_ms = (t_enq - t0) * 1e3 / args.steps
    # the same loop with the copies alone: what the host link allows this step
    for i in range(args.warmup):
        e2e_step(i, compute=False)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        e2e_step(i, compute=False)
    torch.cuda.synchronize()
    copies_ms = (time.perf_counter() - t0) * 1e3 / args.steps
    e2e_value = whole_job_tops(world, e2e_ms)

    cpu = None
    if rank == 0 and world == 1:
        # whole steps (every row of both shapes) until about 10 s of CPU work
        rows = tuple(cc.M for cc in cases)
        ops = secs = 0.0
        reps = 0
        while reps < 6 and (reps == 0 or secs < 10.0):
            o, s_, threads = oracle_sample(rows, 31 * reps)
            ops += o
            secs += s_
            reps += 1
        cpu = {"value": ops / secs / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{reps} whole steps (all {rows[0]} + {rows[1]} token rows of the two "
                         f"shapes); weights quantized outside the timed part",
               "seconds": secs}
        # the same oracle on one host thread, over a smaller sample
        import oracle
        oracle.set_num_threads(1)
        try:
            rows1 = (64, 32)
            o1, s1, _ = oracle_sample(rows1, 977)
        finally:
            oracle.set_num_threads(threads)
        cpu["single_thread"] = {"value": o1 / s1 / 1e12, "unit": UNIT, "cores": 1,
                                "sample": f"{rows1[0]} + {rows1[1]} token rows of the two shapes",
                                "seconds": s1}
        if not args.no_oracle_configs:
            cpu["other_workloads"], _ = oracle_configs_sample()

    if dist:
        dist.destroy_process_group()
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": WORKLOAD, "shapes_MKN": [[cc.M, cc.K, cc.N] for cc in cases],
                   "group": 128, "weights": "GEMM-resident fp16-held INT8 codes",
                   "l2": f"{N_SETS} rotating input sets (~{N_SETS * 125} MB) > 129 MB L2",
                   "launch": "one CUDA graph per input set, replayed per step",
                   "parallelism": f"replicas x{world}"},
        "gpu_launches": launches_per_step * args.steps,
        "overlap": {"ms_per_step": overlap_ms, "value": whole_job_tops(world, overlap_ms),
                    "how": "the same step captured with ck_set_launch_overlap(1), rank 0"},
        "roofline": roofline,
        "gemm_small": gemm_small,
        "int8_dense_peak": {"tops": int8_peak, "how": "mma.sync m16n8k32 s8 rate measured live",
                            "frac": value / world / int8_peak},
        "engine_peak": {"tflops": engine_peak, "frac": achieved_tf / engine_peak,
                        "how": "issue rate of tcgen05.mma kind::f16 128x256x16 from shared memory "
                               "on every SM, measured live (ck_measure_tcgen05_f16_tflops); frac "
                               "= the 4096^3 GEMM alone against it"},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "host_enqueue_ms_per_step": enqueue_ms,
                "copies_only_ms_per_step": copies_ms,
                "how": "ck_int8_linear (C ABI) per step with pinned host->device copies of x "
                       "and device->host copies of y in the timed region (host wall clock), "
                       f"{NB} buffers on three streams"},
        "cpu_baseline": cpu,
        "clocks": clock_info,
        "gemv": gemv,
        "gemv_lowbit": gemv_lowbit,
        "quantize": quantize,
        "enqueue": enqueue,
        "swiglu_mlp": mlp,
        "dit_pass": dit,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world, rank, local = dist_env()
    if args.case:
        run_case(args)
    elif args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
