"""Small-M GEMV over the GEMV-resident layout: the relayout is byte-exact
against the oracle's pack on the same codes, and the GEMV output matches the
oracle's linear (bf16 rel L2 <= 2e-3) and, bit for bit, the GEMM path's
ck_int8_linear (same exact int32 sums and the same f32 dequant)."""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_group_gb300 as ck
from swiglu_mlp_group_gb300 import workloads as wl

from gpu_helpers import assert_output_close, device, poll_ok

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,K", [(16, 32), (40, 256), (128, 4096), (4104, 3072)])
def test_pack_matches_oracle_bytes(N, K):
    dev = device()
    g = torch.Generator().manual_seed(N + K)
    Wq = torch.randint(-127, 128, (N, K), generator=g, dtype=torch.int32).to(torch.int8)
    sw = torch.rand(N, generator=g) + 0.1
    packed = ck.prepare_weight(Wq.to(dev), sw.to(dev), ck.CK_WLAYOUT_GEMV_PACKED)
    ref = oracle.pack_gemv(Wq.numpy(), sw.numpy())
    np.testing.assert_array_equal(packed.cpu().numpy(), ref)
    poll_ok()


def _gemv_case(M, N, K, g, seed, bias=False, act="none"):
    dev = device()
    Kin = 2 * K if act == "swiglu" else K
    x = wl.activation(M, Kin, seed, 0.005, 30.0)
    W = wl.weight(N, K, seed + 1)
    b = wl.bias(N, seed + 2) if bias else None
    Wq, sw = ck.quantize_weight(W.to(dev), g)
    Wp = ck.prepare_weight(Wq, sw, ck.CK_WLAYOUT_GEMV_PACKED)
    bd = None if b is None else b.to(dev)
    y = ck.gemv_smallM(x.to(dev), Wp, N, g, bias=bd, act=act)
    y_lin = ck.int8_linear(x.to(dev), Wq, sw, g, bias=bd, act=act)
    poll_ok()
    if b is None:
        assert torch.equal(y, y_lin)  # same exact sums, same dequant arithmetic
    else:
        assert_output_close(y, wl.bf16_bits(y_lin.cpu()))
    Wq_o, sw_o = oracle.quantize_weight(W.numpy(), g)
    y_o = oracle.int8_linear(wl.bf16_bits(x), Wq_o, sw_o, g,
                             None if b is None else wl.bf16_bits(b), act)
    return assert_output_close(y, y_o)


@pytest.mark.parametrize("M", [1, 2, 4, 8])
@pytest.mark.parametrize("N,K", [(12288, 4096), (4096, 12288), (18432, 3072)])
def test_gemv_workload_shapes(M, N, K):
    _gemv_case(M, N, K, 128, seed=600 + M + K)


@pytest.mark.parametrize("M", [1, 3, 7])
def test_gemv_ragged_with_bias(M):
    _gemv_case(M, 40, 256, 64, seed=700 + M, bias=True)


def test_gemv_swiglu_input():
    _gemv_case(5, 264, 512, 128, seed=800, act="swiglu")


def test_gemv_dequant_on_shared_codes_equals_full_call():
    dev = device()
    M, N, K, g = 4, 4096, 3072, 128
    x = wl.activation(M, K, 901).to(dev)
    Wq, sw = ck.quantize_weight(wl.weight(N, K, 902).to(dev), g)
    Wp = ck.prepare_weight(Wq, sw, ck.CK_WLAYOUT_GEMV_PACKED)
    xq, sx = ck.rotate_quantize_act(x, g)
    y1 = ck.int8_gemv_dequant(xq, sx, Wp, N)
    y2 = ck.gemv_smallM(x, Wp, N, g)
    poll_ok()
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("M,N,K", [(1, 512, 16384), (3, 264, 32768), (8, 520, 16384)])
def test_gemv_long_rows(M, N, K):
    # K > 12288: the activation fragments are read through L1 instead of being
    # staged in shared memory; covers the dp4a (M <= 4) and MMA (M > 4) engines
    _gemv_case(M, N, K, 128, seed=1000 + M + K)


@pytest.mark.parametrize("M", [5, 6])
def test_gemv_mma_engine_ragged_tokens(M):
    _gemv_case(M, 1000, 1024, 64, seed=1100 + M, bias=True)


@pytest.mark.parametrize("M", [1, 2, 5])
def test_gemv_residual_and_in_place(M):
    # both engines (dp4a for one or two tokens, the MMA beyond), in place too
    dev = device()
    N, K, g = 264, 512, 128
    x = wl.activation(M, K, 1200 + M)
    W = wl.weight(N, K, 1201 + M)
    b = wl.bias(N, 1202 + M)
    r = (torch.randn(M, N, generator=torch.Generator().manual_seed(1203 + M)) * 2).to(torch.bfloat16)
    Wq, sw = ck.quantize_weight(W.to(dev), g)
    Wp = ck.prepare_weight(Wq, sw, ck.CK_WLAYOUT_GEMV_PACKED)
    y = ck.gemv_smallM(x.to(dev), Wp, N, g, bias=b.to(dev), residual=r.to(dev))
    y_in = r.to(dev).clone()
    ck.gemv_smallM(x.to(dev), Wp, N, g, bias=b.to(dev), residual=y_in, out=y_in)
    xq, sx = ck.rotate_quantize_act(x.to(dev), g)
    y_dq = ck.int8_gemv_dequant(xq, sx, Wp, N, bias=b.to(dev), residual=r.to(dev))
    poll_ok()
    assert torch.equal(y, y_in) and torch.equal(y, y_dq)
    Wq_o, sw_o = oracle.quantize_weight(W.numpy(), g)
    y_o = oracle.int8_linear(wl.bf16_bits(x), Wq_o, sw_o, g, wl.bf16_bits(b),
                             residual_bits=wl.bf16_bits(r))
    assert_output_close(y, y_o)


# Shapes where every CTA quantizes the activation rows itself (one kernel):
# M * round_up(K / 32, 32) <= 512, K <= 12288; K / 32 not a multiple of 32
# leaves idle lanes in the last warp of a row's team.
@pytest.mark.parametrize("g", [64, 128, 256])
@pytest.mark.parametrize("act", ["none", "swiglu"])
@pytest.mark.parametrize("M,N,K", [(1, 1032, 12288), (2, 264, 4096), (3, 520, 4864),
                                   (5, 40, 256), (7, 136, 1792), (8, 2056, 2048)])
def test_in_cta_quantizer_matches_the_two_kernel_path(g, act, M, N, K):
    dev = device()
    Kin = 2 * K if act == "swiglu" else K
    x = wl.activation(M, Kin, 1000 + M + K, 0.005, 30.0).to(dev)
    Wq, sw = ck.quantize_weight(wl.weight(N, K, 1001 + K).to(dev), g)
    Wp = ck.prepare_weight(Wq, sw, ck.CK_WLAYOUT_GEMV_PACKED)
    b = wl.bias(N, 1002).to(dev)
    res = wl.activation(M, N, 1003).to(dev)
    ws = torch.full((ck.workspace_bytes(ck.CK_OP_GEMV_SMALLM, M, K, N),), 0x5A, dtype=torch.uint8,
                    device=dev)
    try:
        ck.debug_force_gemv_quantizer(2)
        y = ck.gemv_smallM(x, Wp, N, g, bias=b, act=act, workspace=ws, residual=res)
        torch.cuda.synchronize()
        assert bool((ws == 0x5A).all())  # the one-kernel path needs no workspace
        ck.debug_force_gemv_quantizer(1)
        y_pair = ck.gemv_smallM(x, Wp, N, g, bias=b, act=act, workspace=ws, residual=res)
    finally:
        ck.debug_force_gemv_quantizer(0)
    xq, sx = ck.rotate_quantize_act(x, g, act=act, K=K)
    y_two = ck.int8_gemv_dequant(xq, sx, Wp, N, bias=b, residual=res)
    poll_ok()
    assert torch.equal(y.view(torch.int16), y_two.view(torch.int16))
    assert torch.equal(y_pair.view(torch.int16), y_two.view(torch.int16))


def test_in_cta_quantizer_against_the_oracle():
    try:
        ck.debug_force_gemv_quantizer(2)
        _gemv_case(3, 520, 4864, 256, seed=1100, bias=True, act="swiglu")
        _gemv_case(8, 2056, 2048, 64, seed=1101, bias=True)
    finally:
        ck.debug_force_gemv_quantizer(0)
