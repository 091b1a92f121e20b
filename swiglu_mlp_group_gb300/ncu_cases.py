"""Small, self-contained runs of single kernels for Nsight Compute captures.

    python -m swiglu_mlp_group_gb300.ncu_cases <case> [--reps N]

Each case builds its inputs (seeded, synthetic), runs its kernels a few times
and exits; device memory stays well under a few GB so a capture of one launch
ends by itself.  Cases:
  linear_4096   ConvRot linear at M = K = N = 4096 (quantize + GEMM launches)
  gemm_4096     the GEMM alone on pre-quantized codes, M = K = N = 4096
  gateup_4096   the packed gate|up linear of the MLP, M=4096, K=3072, N=24576
  quant_4096    the activation quantizer alone, M = K = 4096
  swiglu_4096   the swiglu activation quantizer, M=4096, I=12288
  gemv_<M>      small-M GEMV over the packed layout, N=12288, K=4096
"""
from __future__ import annotations

import argparse
import sys

import torch

import swiglu_mlp_group_gb300 as ck
from swiglu_mlp_group_gb300 import workloads as wl


def main(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("case")
    p.add_argument("--reps", type=int, default=3)
    a = p.parse_args(argv)
    ck.build()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    g = 128
    if a.case in ("linear_4096", "gemm_4096", "gateup_4096"):
        M, K, N = (4096, 3072, 24576) if a.case == "gateup_4096" else (4096, 4096, 4096)
        x = wl.activation(M, K, 11, 0.005, 30.0).to(dev)
        Wq, sw = ck.quantize_weight(wl.weight(N, K, 12).to(dev), g)
        W16 = ck.prepare_weight(Wq, sw, ck.CK_WLAYOUT_GEMM_F16)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        if a.case == "gemm_4096":
            xq16, sx = ck.rotate_quantize_act_f16(x, g)
            for _ in range(a.reps):
                ck.int8_gemm_dequant(xq16, sx, W16, sw, out=y)
        else:
            for _ in range(a.reps):
                ck.int8_linear(x, W16, sw, g, wlayout=ck.CK_WLAYOUT_GEMM_F16, out=y)
    elif a.case == "quant_4096":
        x = wl.activation(4096, 4096, 13, 0.005, 30.0).to(dev)
        for _ in range(a.reps):
            ck.rotate_quantize_act_f16(x, g)
    elif a.case == "swiglu_4096":
        h = wl.activation(4096, 2 * 12288, 14).to(dev)
        for _ in range(a.reps):
            ck.rotate_quantize_act_f16(h, g, act="swiglu")
    elif a.case.startswith("gemv_"):
        M = int(a.case.split("_")[1])
        N, K = 12288, 4096
        x = wl.activation(M, K, 15).to(dev)
        Wq, sw = ck.quantize_weight(wl.weight(N, K, 16).to(dev), g)
        Wp = ck.prepare_weight(Wq, sw, ck.CK_WLAYOUT_GEMV_PACKED)
        for _ in range(a.reps):
            ck.gemv_smallM(x, Wp, N, g)
    else:
        raise SystemExit(f"unknown case {a.case}")
    torch.cuda.synchronize()
    if ck.poll_device_status() != ck.CK_OK:
        raise SystemExit("a device-side wait timed out")
    return 0


if __name__ == "__main__":
    sys.exit(main())
