"""End-to-end parity of the ConvRot W8A8 linear (GPU weight quantization, GPU
activation quantization, tcgen05 GEMM, fused dequant) with the oracle: bf16
output relative L2 <= 2e-3, on the workloads' shapes.  The two large shapes are
checked on sampled token rows (rows are independent: per-token scales), in the
same launch configuration the benchmark times."""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_group_gb300 as ck
from swiglu_mlp_group_gb300 import workloads as wl

from gpu_helpers import (WEIGHT_CODE_MISMATCH_FRACTION, assert_codes_match, assert_output_close,
                         device, poll_ok)

pytestmark = pytest.mark.gpu


def _run_case(c, wlayout, rows=None, M=None):
    dev = device()
    x = c.x() if M is None else wl.activation(M, c.K, 1000 * c.seed + 9, c.outlier_frac,
                                              c.outlier_scale)
    W, b = c.W(), c.b()
    Wq, sw = ck.quantize_weight(W.to(dev), c.g)
    Wdev = Wq if wlayout == ck.CK_WLAYOUT_ROWMAJOR_I8 else ck.prepare_weight(Wq, sw, wlayout)
    y = ck.int8_linear(x.to(dev), Wdev, sw, c.g, bias=None if b is None else b.to(dev),
                       wlayout=wlayout, N=c.N)
    poll_ok()
    Wq_o, sw_o = oracle.quantize_weight(W.numpy(), c.g)
    assert_codes_match(Wq.cpu().numpy(), Wq_o, "weight codes", WEIGHT_CODE_MISMATCH_FRACTION)
    xb = wl.bf16_bits(x)
    bb = None if b is None else wl.bf16_bits(b)
    if rows is not None:
        xb = xb[rows]
        y = y[torch.as_tensor(rows, device=dev)]
    y_o = oracle.int8_linear(xb, Wq_o, sw_o, c.g, bb)
    return assert_output_close(y, y_o)


@pytest.mark.parametrize("wlayout", [ck.CK_WLAYOUT_ROWMAJOR_I8, ck.CK_WLAYOUT_GEMM_F16])
def test_linear_tiny_with_bias(wlayout):
    _run_case(wl.LINEAR_TINY, wlayout)


@pytest.mark.parametrize("M", [1, 5, 100, 129, 300])
def test_linear_ragged_token_counts(M):
    _run_case(wl.LINEAR_TINY, ck.CK_WLAYOUT_GEMM_F16, M=M)


def test_linear_2048x3072x1024_full():
    _run_case(wl.LINEAR_2048, ck.CK_WLAYOUT_GEMM_F16)


def test_linear_4096_cubed_sampled_rows():
    rows = np.sort(np.random.default_rng(5).choice(4096, 256, replace=False))
    rows[-1] = 4095
    _run_case(wl.LINEAR_4096, ck.CK_WLAYOUT_GEMM_F16, rows=rows)


@pytest.mark.parametrize("N,n_rows", [(9216, 128), (3072, 256)])
def test_dit_block_linears_sampled_rows(N, n_rows):
    # the DiT-shaped pass's qkv (3072 -> 9216) and attention-out (3072 -> 3072)
    # linears at M = 4096 tokens, N(0, 1) activations, no bias, in the launch
    # configuration the benchmark times; checked on sampled rows (the first and
    # last included)
    case = wl.LinearCase(f"dit_linear_4096x3072x{N}_g128", 4096, 3072, N, 128, 40 + N % 7, 0.0,
                         1.0, False)
    rows = np.sort(np.random.default_rng(N).choice(np.arange(1, 4095), n_rows - 2, replace=False))
    rows = np.concatenate([[0], rows, [4095]])
    _run_case(case, ck.CK_WLAYOUT_GEMM_F16, rows=rows)


def test_linear_error_vs_fp32_is_int8_noise():
    # the pages report ~0.9% relative error of the INT8 path against float32
    dev = device()
    c = wl.LINEAR_2048
    x, W = c.x(), c.W()
    Wq, sw = ck.quantize_weight(W.to(dev), c.g)
    y = ck.int8_linear(x.to(dev), Wq, sw, c.g)
    rows = np.arange(0, 2048, 16)
    y_ref = oracle.reference_linear_f64(x.float().numpy()[rows], W.numpy())
    err = oracle.rel_l2(y.float().cpu().numpy()[rows], y_ref)
    assert 1e-3 < err < 3e-2


def test_linear_swiglu_input_act():
    dev = device()
    M, I, N, g = 96, 512, 256, 128
    h = wl.activation(M, 2 * I, seed=41)
    W = wl.weight(N, I, seed=42)
    Wq, sw = ck.quantize_weight(W.to(dev), g)
    y = ck.int8_linear(h.to(dev), Wq, sw, g, act="swiglu")
    Wq_o, sw_o = oracle.quantize_weight(W.numpy(), g)
    y_o = oracle.int8_linear(wl.bf16_bits(h), Wq_o, sw_o, g, None, "swiglu")
    assert_output_close(y, y_o)


@pytest.mark.parametrize("tile", [64, 128, 256, 512, 448, 2128])
def test_linear_with_bias_on_every_gemm_variant(tile):
    # the fused dequant + bias epilogue of each GEMM variant, ragged M and N
    dev = device()
    M, K, N, g = 300, 1024, 520, 128
    x = wl.activation(M, K, 61, 0.005, 30.0)
    W = wl.weight(N, K, 62)
    b = wl.bias(N, 63)
    Wq, sw = ck.quantize_weight(W.to(dev), g)
    W16 = ck.prepare_weight(Wq, sw, ck.CK_WLAYOUT_GEMM_F16)
    ck.debug_force_gemm_tile(tile)
    try:
        y = ck.int8_linear(x.to(dev), W16, sw, g, bias=b.to(dev), wlayout=ck.CK_WLAYOUT_GEMM_F16)
        poll_ok()
    finally:
        ck.debug_force_gemm_tile(0)
    Wq_o, sw_o = oracle.quantize_weight(W.numpy(), g)
    assert_output_close(y, oracle.int8_linear(wl.bf16_bits(x), Wq_o, sw_o, g, wl.bf16_bits(b)))


def test_linear_maximum_k():
    # K = 32768, the largest accepted row: the quantizer's two-units-per-thread
    # path and a 32-chunk exact-int32 GEMM
    dev = device()
    M, K, N, g = 24, 32768, 264, 256
    x = wl.activation(M, K, 71, 0.005, 30.0)
    W = wl.weight(N, K, 72)
    Wq, sw = ck.quantize_weight(W.to(dev), g)
    y = ck.int8_linear(x.to(dev), Wq, sw, g, N=N)
    poll_ok()
    Wq_o, sw_o = oracle.quantize_weight(W.numpy(), g)
    assert_codes_match(Wq.cpu().numpy(), Wq_o, "weight codes", WEIGHT_CODE_MISMATCH_FRACTION)
    assert_output_close(y, oracle.int8_linear(wl.bf16_bits(x), Wq_o, sw_o, g))


@pytest.mark.parametrize("tile", [0, 256, 448])
def test_linear_residual_and_in_place(tile):
    # y = linear(x) + bias + residual, the residual added in the epilogue before
    # the one rounding (comfy-kitchen PR #248, Commits); in place (residual is
    # y) gives the same bits; both GEMM variants
    dev = device()
    M, K, N, g = 300, 1024, 520, 128
    x = wl.activation(M, K, 81, 0.005, 30.0)
    W = wl.weight(N, K, 82)
    b = wl.bias(N, 83)
    r = (torch.randn(M, N, generator=torch.Generator().manual_seed(84)) * 4).to(torch.bfloat16)
    Wq, sw = ck.quantize_weight(W.to(dev), g)
    W16 = ck.prepare_weight(Wq, sw, ck.CK_WLAYOUT_GEMM_F16)
    ck.debug_force_gemm_tile(tile)
    try:
        rd = r.to(dev)
        y = ck.int8_linear(x.to(dev), W16, sw, g, bias=b.to(dev), residual=rd,
                           wlayout=ck.CK_WLAYOUT_GEMM_F16)
        y_in = rd.clone()
        ck.int8_linear(x.to(dev), W16, sw, g, bias=b.to(dev), residual=y_in, out=y_in,
                       wlayout=ck.CK_WLAYOUT_GEMM_F16)
        poll_ok()
    finally:
        ck.debug_force_gemm_tile(0)
    assert torch.equal(y, y_in)
    Wq_o, sw_o = oracle.quantize_weight(W.numpy(), g)
    y_o = oracle.int8_linear(wl.bf16_bits(x), Wq_o, sw_o, g, wl.bf16_bits(b),
                             residual_bits=wl.bf16_bits(r))
    assert_output_close(y, y_o)


def test_gemm_dequant_residual_is_added_once():
    # the same codes with and without a residual: the difference is the residual
    # up to one bf16 rounding of the sum
    dev = device()
    M, K, N, g = 128, 512, 256, 64
    x = wl.activation(M, K, 91).to(dev)
    Wq, sw = ck.quantize_weight(wl.weight(N, K, 92).to(dev), g)
    W16 = ck.prepare_weight(Wq, sw, ck.CK_WLAYOUT_GEMM_F16)
    xq16, sx = ck.rotate_quantize_act_f16(x, g)
    r = torch.full((M, N), 0.25, dtype=torch.bfloat16, device=dev)
    y0 = ck.int8_gemm_dequant(xq16, sx, W16, sw)
    y1 = ck.int8_gemm_dequant(xq16, sx, W16, sw, residual=r)
    poll_ok()
    # y0 and y1 are each rounded once to bf16 (half an ulp: <= 2^-8 relative)
    d = (y1.float() - y0.float() - 0.25).abs()
    bound = (y0.float().abs() + y1.float().abs()) * 2.0 ** -8 + 1e-6
    assert bool((d <= bound).all())
