"""Fused SwiGLU MLP: parity with the oracle (bf16 rel L2 <= 2e-3) of both its
results -- the packed gate|up linear's output h, read from the call's
workspace, and the MLP's output y -- and the accuracy claim of the SwiGLU
page: the fused path's error against an unquantized float reference is no
worse than the staged path that rounds silu(gate) * up to bf16, at the page's
(2048, 3072 -> 1024) shape and the hidden-3072 / intermediate-12288 shape."""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_group_gb300 as ck
from swiglu_mlp_group_gb300 import workloads as wl

from gpu_helpers import assert_output_close, device, poll_ok

pytestmark = pytest.mark.gpu


def _mlp(case, rows=None, wlayout=ck.CK_WLAYOUT_GEMM_F16, with_bias=False):
    dev = device()
    x = case.x()
    Wg, Wu, Wd = case.W_gate(), case.W_up(), case.W_down()
    Wgu = torch.cat([Wg, Wu], 0)
    bgu = wl.bias(2 * case.I, 77) if with_bias else None
    bd = wl.bias(case.H, 78) if with_bias else None
    Wgu_q, sgu = ck.quantize_weight(Wgu.to(dev), case.g)
    Wd_q, sd = ck.quantize_weight(Wd.to(dev), case.g)
    if wlayout == ck.CK_WLAYOUT_GEMM_F16:
        Wgu_dev = ck.prepare_weight(Wgu_q, sgu, wlayout)
        Wd_dev = ck.prepare_weight(Wd_q, sd, wlayout)
    else:
        Wgu_dev, Wd_dev = Wgu_q, Wd_q
    ws = torch.empty(ck.workspace_bytes(ck.CK_OP_SWIGLU_MLP, case.M, case.H, case.I, wlayout),
                     dtype=torch.uint8, device=dev)
    y = ck.swiglu_mlp(x.to(dev), Wgu_dev, sgu, Wd_dev, sd, case.g,
                      bgu=None if bgu is None else bgu.to(dev),
                      bd=None if bd is None else bd.to(dev), wlayout=wlayout, workspace=ws)
    poll_ok()
    # h, the packed gate|up output, where the workspace layout of include/ck.h
    # places it: after the fp16-held codes of x (2 M H bytes) and their scales
    # (4 M bytes), each rounded up to 256 bytes
    up = lambda v: (v + 255) // 256 * 256
    h_off = up(2 * case.M * case.H) + up(4 * case.M)
    h = ws[h_off:h_off + case.M * 2 * case.I * 2].view(torch.bfloat16).view(case.M, 2 * case.I)
    Wgu_o, sgu_o = oracle.quantize_weight(Wgu.numpy(), case.g)
    Wd_o, sd_o = oracle.quantize_weight(Wd.numpy(), case.g)
    xb = wl.bf16_bits(x)
    if rows is not None:
        xb = xb[rows]
        y = y[torch.as_tensor(rows, device=dev)]
        h = h[torch.as_tensor(rows, device=dev)]
    bgu_b = None if bgu is None else wl.bf16_bits(bgu)
    bd_b = None if bd is None else wl.bf16_bits(bd)
    assert_output_close(h, oracle.int8_linear(xb, Wgu_o, sgu_o, case.g, bgu_b), "h (gate|up)")
    y_o, _ = oracle.swiglu_mlp(xb, Wgu_o, sgu_o, bgu_b, Wd_o, sd_o, bd_b, case.g)
    assert_output_close(y, y_o)
    return y, (xb, Wg, Wu, Wd, Wgu_o, sgu_o, Wd_o, sd_o)


def test_mlp_small_with_bias_both_layouts():
    case = wl.MlpCase("small", 64, 256, 128, 64, 8, 0.01, 20.0)
    _mlp(case, with_bias=True, wlayout=ck.CK_WLAYOUT_ROWMAJOR_I8)
    _mlp(case, with_bias=True, wlayout=ck.CK_WLAYOUT_GEMM_F16)


def _fused_vs_staged(case, rows):
    y, (xb, Wg, Wu, Wd, Wgu_o, sgu_o, Wd_o, sd_o) = _mlp(case, rows=rows)
    ref = oracle.reference_mlp_f64(oracle.bf16_bits_to_f32(xb), Wg.numpy(), Wu.numpy(), Wd.numpy())
    e_fused = oracle.rel_l2(y.float().cpu().numpy(), ref)
    staged = oracle.staged_swiglu_mlp(xb, Wgu_o, sgu_o, None, Wd_o, sd_o, None, case.g)
    e_staged = oracle.rel_l2(oracle.bf16_bits_to_f32(staged), ref)
    assert e_fused <= e_staged, (e_fused, e_staged)
    return e_fused, e_staged


def test_mlp_2048_h3072_i1024_full_and_fused_no_worse_than_staged():
    _fused_vs_staged(wl.MLP_2048, rows=None)


def test_mlp_4096_h3072_i12288_sampled_rows_and_fused_no_worse_than_staged():
    rows = np.sort(np.random.default_rng(6).choice(4096, 256, replace=False))
    _fused_vs_staged(wl.MLP_4096, rows=rows)


def test_mlp_residual_on_the_down_linear():
    # the block's skip connection fused into the down linear's epilogue
    dev = device()
    M, H, I, g = 96, 512, 1024, 128
    x = wl.activation(M, H, 301)
    Wgu = torch.cat([wl.weight(I, H, 302), wl.weight(I, H, 303)], 0)
    Wd = wl.weight(H, I, 304)
    Wgu_q, sgu = ck.quantize_weight(Wgu.to(dev), g)
    Wd_q, sd = ck.quantize_weight(Wd.to(dev), g)
    Wgu16 = ck.prepare_weight(Wgu_q, sgu, ck.CK_WLAYOUT_GEMM_F16)
    Wd16 = ck.prepare_weight(Wd_q, sd, ck.CK_WLAYOUT_GEMM_F16)
    xd = x.to(dev)
    y = ck.swiglu_mlp(xd, Wgu16, sgu, Wd16, sd, g, residual=xd, wlayout=ck.CK_WLAYOUT_GEMM_F16)
    poll_ok()
    Wgu_o, sgu_o = oracle.quantize_weight(Wgu.numpy(), g)
    Wd_o, sd_o = oracle.quantize_weight(Wd.numpy(), g)
    y_o, _ = oracle.swiglu_mlp(wl.bf16_bits(x), Wgu_o, sgu_o, None, Wd_o, sd_o, None, g,
                               residual_bits=wl.bf16_bits(x))
    assert_output_close(y, y_o)
