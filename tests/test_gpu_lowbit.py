"""W6A8 / W4A8 decode weights on the GPU (comfy-kitchen PR #248, "Performance
improvements for qwen 3.x (Part 2)", Commits and Description: 4- and 6-bit
weight decode rounded onto the INT8 grid): the b-bit weight quantizer against
the oracle's codes and scales, the low-bit relayout byte for byte against the
oracle's pack, and the GEMV over it against the oracle's linear on the same
codes (bf16 rel L2 <= 2e-3) and, bit for bit, against the INT8-layout GEMV on
those codes (the sums are 2^(8-b) times as large and the row scale 2^(8-b)
times smaller: every rounding is the same)."""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_group_gb300 as ck
from swiglu_mlp_group_gb300 import workloads as wl

from gpu_helpers import (WEIGHT_CODE_MISMATCH_FRACTION, assert_codes_match, assert_output_close,
                         assert_scales_match, device, poll_ok)

pytestmark = pytest.mark.gpu

LAYOUT = {8: ck.CK_WLAYOUT_GEMV_PACKED, 6: ck.CK_WLAYOUT_GEMV_PACKED_W6,
          4: ck.CK_WLAYOUT_GEMV_PACKED_W4}


@pytest.mark.parametrize("bits", [4, 6, 8])
@pytest.mark.parametrize("N,K,g", [(40, 256, 64), (264, 3072, 128), (1032, 4096, 256)])
def test_weight_quantizer_bits_matches_oracle(bits, N, K, g):
    dev = device()
    W = wl.weight(N, K, 2000 + bits + K)
    Wq, sw = ck.quantize_weight_bits(W.to(dev), g, bits)
    poll_ok()
    Wq_o, sw_o = oracle.quantize_weight_bits(W.numpy(), g, bits)
    qmax = (1 << (bits - 1)) - 1
    assert int(Wq.abs().max()) <= qmax
    assert_codes_match(Wq.cpu().numpy(), Wq_o, f"{bits}-bit weight codes",
                       WEIGHT_CODE_MISMATCH_FRACTION)
    assert_scales_match(sw.cpu().numpy(), sw_o, f"{bits}-bit weight scales")
    if bits == 8:
        Wq8, sw8 = ck.quantize_weight(W.to(dev), g)
        assert torch.equal(Wq8, Wq) and torch.equal(sw8, sw)


@pytest.mark.parametrize("bits", [4, 6])
@pytest.mark.parametrize("N,K", [(16, 32), (40, 256), (4104, 3072)])
def test_pack_lowbit_matches_oracle_bytes(bits, N, K):
    dev = device()
    qmax = (1 << (bits - 1)) - 1
    g = torch.Generator().manual_seed(3000 + N + K + bits)
    Wq = torch.randint(-qmax, qmax + 1, (N, K), generator=g, dtype=torch.int32).to(torch.int8)
    sw = torch.rand(N, generator=g) + 0.1
    packed = ck.prepare_weight(Wq.to(dev), sw.to(dev), LAYOUT[bits])
    poll_ok()
    np.testing.assert_array_equal(packed.cpu().numpy(),
                                  oracle.pack_gemv_lowbit(Wq.numpy(), sw.numpy(), bits))


def _lowbit_case(bits, M, N, K, g, seed, bias=False, act="none", residual=False):
    dev = device()
    Kin = 2 * K if act == "swiglu" else K
    x = wl.activation(M, Kin, seed, 0.005, 30.0)
    W = wl.weight(N, K, seed + 1)
    b = wl.bias(N, seed + 2) if bias else None
    r = (torch.randn(M, N, generator=torch.Generator().manual_seed(seed + 3)) * 2).to(
        torch.bfloat16) if residual else None
    bd = None if b is None else b.to(dev)
    rd = None if r is None else r.to(dev)
    Wq, sw = ck.quantize_weight_bits(W.to(dev), g, bits)
    Wp = ck.prepare_weight(Wq, sw, LAYOUT[bits])
    y = ck.gemv_smallM(x.to(dev), Wp, N, g, bias=bd, act=act, residual=rd, wlayout=LAYOUT[bits])
    # the same codes in the INT8 layout
    Wp8 = ck.prepare_weight(Wq, sw, ck.CK_WLAYOUT_GEMV_PACKED)
    y8 = ck.gemv_smallM(x.to(dev), Wp8, N, g, bias=bd, act=act, residual=rd)
    xq, sx = ck.rotate_quantize_act(x.to(dev), g, act=act, K=K)
    y_dq = ck.packed_gemv_dequant(xq, sx, Wp, LAYOUT[bits], N, bias=bd, residual=rd)
    poll_ok()
    assert torch.equal(y.view(torch.int16), y8.view(torch.int16))
    assert torch.equal(y.view(torch.int16), y_dq.view(torch.int16))
    Wq_o, sw_o = oracle.quantize_weight_bits(W.numpy(), g, bits)
    y_o = oracle.int8_linear(wl.bf16_bits(x), Wq_o, sw_o, g,
                             None if b is None else wl.bf16_bits(b), act,
                             residual_bits=None if r is None else wl.bf16_bits(r))
    return assert_output_close(y, y_o)


@pytest.mark.parametrize("bits", [4, 6])
@pytest.mark.parametrize("M", [1, 2, 4, 8])
@pytest.mark.parametrize("N,K", [(12288, 4096), (4096, 12288), (18432, 3072)])
def test_lowbit_gemv_workload_shapes(bits, M, N, K):
    _lowbit_case(bits, M, N, K, 128, seed=3100 + M + K + bits)


@pytest.mark.parametrize("bits", [4, 6])
@pytest.mark.parametrize("M", [1, 3, 7])
def test_lowbit_gemv_ragged_with_bias_and_residual(bits, M):
    _lowbit_case(bits, M, 40, 256, 64, seed=3200 + M + bits, bias=True, residual=True)


@pytest.mark.parametrize("bits", [4, 6])
def test_lowbit_gemv_swiglu_input(bits):
    _lowbit_case(bits, 5, 264, 512, 128, seed=3300 + bits, act="swiglu", bias=True)


@pytest.mark.parametrize("bits", [4, 6])
@pytest.mark.parametrize("M,N,K", [(1, 512, 16384), (8, 520, 16384)])
def test_lowbit_gemv_long_rows(bits, M, N, K):
    # activation fragments read through L1 instead of shared memory
    _lowbit_case(bits, M, N, K, 128, seed=3400 + M + bits)


@pytest.mark.parametrize("bits", [4, 6])
@pytest.mark.parametrize("act", ["none", "swiglu"])
@pytest.mark.parametrize("M,N,K,g", [(1, 1032, 12288, 128), (2, 264, 4096, 64),
                                     (8, 2056, 2048, 256)])
def test_lowbit_in_cta_quantizer_matches_the_two_kernel_path(bits, act, M, N, K, g):
    dev = device()
    Kin = 2 * K if act == "swiglu" else K
    x = wl.activation(M, Kin, 3500 + M + K, 0.005, 30.0).to(dev)
    Wq, sw = ck.quantize_weight_bits(wl.weight(N, K, 3501 + K).to(dev), g, bits)
    Wp = ck.prepare_weight(Wq, sw, LAYOUT[bits])
    b = wl.bias(N, 3502).to(dev)
    try:
        ck.debug_force_gemv_quantizer(2)
        y = ck.gemv_smallM(x, Wp, N, g, bias=b, act=act, wlayout=LAYOUT[bits])
        ck.debug_force_gemv_quantizer(1)
        y_two = ck.gemv_smallM(x, Wp, N, g, bias=b, act=act, wlayout=LAYOUT[bits])
    finally:
        ck.debug_force_gemv_quantizer(0)
    poll_ok()
    assert torch.equal(y.view(torch.int16), y_two.view(torch.int16))


@pytest.mark.parametrize("bits", [4, 6, 8])
@pytest.mark.parametrize("M,N,K", [(1, 24, 64), (3, 40, 128), (8, 16, 192), (2, 520, 448)])
def test_lowbit_gemv_short_rows(bits, M, N, K):
    # K / 32 below the 16 warps of a CTA: fewer K-slices than warps, the rest idle
    _lowbit_case(bits, M, N, K, 64, seed=3600 + M + K + bits, bias=True)


@pytest.mark.parametrize("bits", [4, 6])
def test_weight_quantizer_bits_degenerate_rows(bits):
    # a zero row (scale 0, codes 0), a constant row, one huge and one tiny row
    dev = device()
    N, K, g = 8, 256, 64
    W = wl.weight(N, K, 3700 + bits)
    W[0] = 0.0
    W[1] = 0.75
    W[2] *= 1e30
    W[3] *= 1e-30
    Wq, sw = ck.quantize_weight_bits(W.to(dev), g, bits)
    poll_ok()
    Wq_o, sw_o = oracle.quantize_weight_bits(W.numpy(), g, bits)
    assert float(sw[0]) == 0.0 and not bool(Wq[0].any())
    assert_codes_match(Wq.cpu().numpy(), Wq_o, f"{bits}-bit weight codes", WEIGHT_CODE_MISMATCH_FRACTION)
    assert_scales_match(sw.cpu().numpy(), sw_o, f"{bits}-bit weight scales")
