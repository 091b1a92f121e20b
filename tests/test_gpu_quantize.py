"""Parity of the rotate+quantize kernel (weights and activations, act none and
swiglu) with the oracle: codes equal up to +-1 at ties on <= 1e-4 of the
elements, scales within 1e-6 relative."""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_group_gb300 as ck
from swiglu_mlp_group_gb300 import workloads as wl

from gpu_helpers import (WEIGHT_CODE_MISMATCH_FRACTION, assert_codes_match, assert_scales_match,
                         device, poll_ok)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("g,M,K", [(64, 64, 256), (128, 2048, 3072), (256, 33, 512),
                                   (128, 7, 12288), (64, 5, 320), (128, 1, 4096),
                                   (256, 300, 1024)])
def test_activation_quantize(g, M, K):
    dev = device()
    x = wl.activation(M, K, seed=100 + M + K, outlier_frac=0.005, outlier_scale=30.0)
    xq, sx = ck.rotate_quantize_act(x.to(dev), g)
    q_ref, s_ref = oracle.rotate_quantize_act(wl.bf16_bits(x), g)
    assert_scales_match(sx.cpu().numpy(), s_ref)
    assert_codes_match(xq.cpu().numpy(), q_ref)
    poll_ok()


@pytest.mark.parametrize("g,M,I", [(64, 64, 128), (128, 512, 1024), (128, 16, 12288),
                                   (256, 9, 768)])
def test_swiglu_activation_quantize(g, M, I):
    dev = device()
    h = wl.activation(M, 2 * I, seed=200 + M + I) 
    xq, sx = ck.rotate_quantize_act(h.to(dev), g, act="swiglu")
    q_ref, s_ref = oracle.rotate_quantize_act(wl.bf16_bits(h), g, "swiglu")
    assert_scales_match(sx.cpu().numpy(), s_ref)
    assert_codes_match(xq.cpu().numpy(), q_ref)


def test_swiglu_reads_a_strided_view():
    # ldx > 2K: the packed [gate | up] rows live inside a wider buffer
    dev = device()
    M, I, g = 32, 256, 128
    buf = wl.activation(M, 2 * I + 64, seed=7)
    xq, sx = ck.rotate_quantize_act(buf.to(dev), g, act="swiglu", K=I)
    q_ref, s_ref = oracle.rotate_quantize_act(wl.bf16_bits(buf[:, :2 * I]), g, "swiglu")
    assert_scales_match(sx.cpu().numpy(), s_ref)
    assert_codes_match(xq.cpu().numpy(), q_ref)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("g,N,K", [(64, 128, 256), (128, 1024, 3072), (256, 40, 1024),
                                   (128, 3072, 12288)])
def test_weight_quantize(dtype, g, N, K):
    dev = device()
    W = wl.weight(N, K, seed=300 + N + K).to(dtype)
    Wq, sw = ck.quantize_weight(W.to(dev), g)
    q_ref, s_ref = oracle.quantize_weight(W.float().numpy(), g)
    np.testing.assert_array_equal(sw.cpu().numpy(), s_ref)
    assert_codes_match(Wq.cpu().numpy(), q_ref, "weight codes", WEIGHT_CODE_MISMATCH_FRACTION)


def test_degenerate_rows():
    dev = device()
    x = wl.activation(6, 256, seed=9).float()
    x[0] = 0.0                # zero row: scale 0, codes 0
    x[1] = 1.5                # constant row: one nonzero per group after rotation
    x[2, 17] = 1000.0         # a single huge outlier
    x[3] = -0.0
    x = x.to(torch.bfloat16)
    xq, sx = ck.rotate_quantize_act(x.to(dev), 64)
    q_ref, s_ref = oracle.rotate_quantize_act(wl.bf16_bits(x), 64)
    assert sx[0].item() == 0.0 and int(xq[0].abs().sum()) == 0
    assert sx[3].item() == 0.0 and int(xq[3].abs().sum()) == 0
    assert_scales_match(sx.cpu().numpy(), s_ref)
    np.testing.assert_array_equal(xq.cpu().numpy(), q_ref)


@pytest.mark.parametrize("act", ["none", "swiglu"])
def test_maximum_k_quantize(act):
    # K = 32768: two 32-element units per thread
    dev = device()
    M, K, g = 5, 32768, 128
    Kin = 2 * K if act == "swiglu" else K
    x = wl.activation(M, Kin, seed=801 if act == "none" else 802, outlier_frac=0.005,
                      outlier_scale=30.0)
    xq, sx = ck.rotate_quantize_act(x.to(dev), g, act=act)
    q_ref, s_ref = oracle.rotate_quantize_act(wl.bf16_bits(x), g, act)
    assert_scales_match(sx.cpu().numpy(), s_ref)
    assert_codes_match(xq.cpu().numpy(), q_ref)
    poll_ok()
