"""The tcgen05 GEMM engine's int32 accumulators are bit-exact against the
oracle's int64 GEMM on the same INT8 codes, including adversarial +-127
operands whose sums exceed 2^24 (exact only because the kernel drains the f32
tensor-core accumulator into int32 every 1024 products, a sum that stays below
2^24 in magnitude)."""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_group_gb300 as ck

from gpu_helpers import device, poll_ok

pytestmark = pytest.mark.gpu


def _codes(rows, K, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(-127, 128, (rows, K), generator=g, dtype=torch.int32).to(torch.int8)


@pytest.mark.parametrize("M,N,K", [(64, 128, 256), (1, 8, 64), (130, 136, 192),
                                   (128, 256, 1024), (300, 520, 576), (2048, 1024, 3072),
                                   (256, 512, 12288), (513, 264, 4160)])
def test_gemm_s32_bit_exact_random(M, N, K):
    dev = device()
    xq, wq = _codes(M, K, M * 7 + K), _codes(N, K, N * 11 + K)
    acc = ck.debug_int8_gemm_s32(xq.to(dev), wq.to(dev)).cpu().numpy()
    ref = oracle.int8_gemm(xq.numpy(), wq.numpy())
    np.testing.assert_array_equal(acc.astype(np.int64), ref)
    poll_ok()


@pytest.mark.parametrize("K", [1024, 4096, 12288])
def test_gemm_s32_bit_exact_adversarial(K):
    dev = device()
    M, N = 128, 256
    xq = torch.full((M, K), 127, dtype=torch.int8)
    wq = torch.full((N, K), 127, dtype=torch.int8)
    xq[1] = -127
    wq[2] = -127
    xq[3, ::2] = -127              # alternating signs: partial sums cancel
    wq[5, K // 2:] = -127          # sum climbs to +K/2*16129 then back to 0
    xq[7, :] = torch.arange(K) % 255 - 127
    acc = ck.debug_int8_gemm_s32(xq.to(dev), wq.to(dev)).cpu().numpy()
    ref = oracle.int8_gemm(xq.numpy(), wq.numpy())
    assert ref[0, 0] == K * 16129
    assert K < 2048 or ref[0, 0] > 2 ** 24
    np.testing.assert_array_equal(acc.astype(np.int64), ref)
    poll_ok()


@pytest.mark.parametrize("bn", [64, 128, 256, 512, 448, 2128, 4512])
@pytest.mark.parametrize("M,N,K", [(300, 520, 4160), (128, 256, 12288), (700, 1032, 1536)])
def test_gemm_s32_every_tile_width(bn, M, N, K):
    dev = device()
    xq, wq = _codes(M, K, M + 3 * K + bn), _codes(N, K, N + 5 * K + bn)
    ck.debug_force_gemm_tile(bn)
    try:
        acc = ck.debug_int8_gemm_s32(xq.to(dev), wq.to(dev)).cpu().numpy()
    finally:
        ck.debug_force_gemm_tile(0)
    np.testing.assert_array_equal(acc.astype(np.int64), oracle.int8_gemm(xq.numpy(), wq.numpy()))
    poll_ok()


@pytest.mark.parametrize("bn", [64, 128, 256, 512, 448, 2128, 4512])
def test_gemm_dequant_epilogue_matches_exact_sums(bn):
    # y = bf16((f32(acc) * sx * sw + bias) + residual) from the exact int32 sums,
    # written by every tile width: ragged M (a last quad of one row) and ragged N
    # (a last tile holding one 8-column piece); plain fp32 reference of the same
    # formula, within one bf16 ulp (the kernel may fuse a multiply-add)
    dev = device()
    M, N, K = 301, 520, 1024
    xq, wq = _codes(M, K, 1200 + bn), _codes(N, K, 1300 + bn)
    g = torch.Generator().manual_seed(1400 + bn)
    sx = torch.rand(M, generator=g) * 1e-3 + 1e-4
    sw = torch.rand(N, generator=g) * 1e-3 + 1e-4
    b = (torch.randn(N, generator=g) * 0.5).to(torch.bfloat16)
    r = (torch.randn(M, N, generator=g) * 2).to(torch.bfloat16)
    acc = torch.from_numpy(oracle.int8_gemm(xq.numpy(), wq.numpy()))
    y_ref = ((acc.double().float() * sx[:, None] * sw[None, :] + b.float()[None, :]) + r.float())
    y_ref = y_ref.to(torch.bfloat16).float()
    xq16, w16 = xq.to(torch.float16).to(dev), wq.to(torch.float16).to(dev)
    ck.debug_force_gemm_tile(bn)
    try:
        y = ck.int8_gemm_dequant(xq16, sx.to(dev), w16, sw.to(dev), bias=b.to(dev),
                                 residual=r.to(dev))
        y_in = r.to(dev)
        ck.int8_gemm_dequant(xq16, sx.to(dev), w16, sw.to(dev), bias=b.to(dev), residual=y_in,
                             out=y_in)
        y_nb = ck.int8_gemm_dequant(xq16, sx.to(dev), w16, sw.to(dev))
        poll_ok()
    finally:
        ck.debug_force_gemm_tile(0)
    assert torch.equal(y, y_in)
    prod = acc.double().float() * sx[:, None] * sw[None, :]

    def within_one_ulp(got, ref, mag):
        # one bf16 ulp of the result, plus a few f32 ulps of the operands for the
        # fused multiply-add when the sum cancels
        ulp = torch.exp2(torch.floor(torch.log2(ref.abs().clamp_min(2.0 ** -100))) - 7)
        d = (got.float().cpu() - ref).abs()
        assert bool((d <= ulp + mag * 2.0 ** -21).all()), f"max excess {(d - ulp).max().item()}"
        assert (d > 0).float().mean().item() < 0.01

    within_one_ulp(y, y_ref, prod.abs() + b.float().abs()[None, :] + r.float().abs())
    within_one_ulp(y_nb, prod.to(torch.bfloat16).float(), prod.abs())


@pytest.mark.parametrize("bn", [64, 128, 256, 512, 448, 2128, 4512])
def test_gemm_s32_several_tiles_per_cta(bn):
    # more tiles than CTAs (or CTA pairs) for every variant, so each CTA's
    # producer and issuer walk k-blocks across tile boundaries; K = 17 k-blocks
    # (a 16-block chunk and a 1-block chunk per tile), ragged M and N.  The
    # exact int32 reference is a float64 matmul (every partial sum < 2^53).
    dev = device()
    M, N, K = 4200, 2008, 1088
    xq, wq = _codes(M, K, 1500 + bn), _codes(N, K, 1600 + bn)
    ck.debug_force_gemm_tile(bn)
    try:
        acc = ck.debug_int8_gemm_s32(xq.to(dev), wq.to(dev))
    finally:
        ck.debug_force_gemm_tile(0)
    poll_ok()
    ref = (xq.to(dev).double() @ wq.to(dev).double().T).to(torch.int64)
    assert torch.equal(acc.to(torch.int64), ref)


@pytest.mark.parametrize("M,N,K", [(2048, 1024, 3072), (1, 24, 128), (257, 1032, 4160), (128, 256, 12288)])
def test_split_k_bit_exact_and_equal_to_the_unsplit_output(M, N, K):
    # K split between two CTA pairs, the halves' int32 sums added on chip:
    # bit-exact sums (an odd number of k-blocks at K = 4160; sums beyond 2^24
    # in each half at K = 12288 with +-127 rows), and the dequantized bf16 output
    # identical to the automatic variant's (same sums, same epilogue arithmetic)
    dev = device()
    xq, wq = _codes(M, K, 1700 + K), _codes(N, K, 1800 + K)
    xq[0] = 127
    wq[0] = 127
    wq[1] = -127
    g = torch.Generator().manual_seed(1900 + M)
    sx = (torch.rand(M, generator=g) * 1e-3 + 1e-4).to(dev)
    sw = (torch.rand(N, generator=g) * 1e-3 + 1e-4).to(dev)
    b = (torch.randn(N, generator=g) * 0.5).to(torch.bfloat16).to(dev)
    r = (torch.randn(M, N, generator=g) * 2).to(torch.bfloat16).to(dev)
    xq16, w16 = xq.to(torch.float16).to(dev), wq.to(torch.float16).to(dev)
    y_auto = ck.int8_gemm_dequant(xq16, sx, w16, sw, bias=b, residual=r)
    ck.debug_force_gemm_tile(4512)
    try:
        acc = ck.debug_int8_gemm_s32(xq.to(dev), wq.to(dev)).cpu().numpy()
        y = ck.int8_gemm_dequant(xq16, sx, w16, sw, bias=b, residual=r)
        poll_ok()
    finally:
        ck.debug_force_gemm_tile(0)
    ref = oracle.int8_gemm(xq.numpy(), wq.numpy())
    assert ref[0, 0] == K * 16129
    np.testing.assert_array_equal(acc.astype(np.int64), ref)
    assert torch.equal(y, y_auto)


def test_split_k_taken_automatically_where_it_pays():
    # 24 tiles of 256 x 256 at K = 12288: the automatic choice splits K (when
    # the GPU holds 24 four-CTA clusters at once, else it takes the pair
    # tiles); either way the exact sums give the same bf16 output as the
    # 128-column pair tiles
    dev = device()
    M, N, K = 512, 3072, 12288
    assert ck.debug_gemm_tile_choice(M, N, K, 152) == 4512
    xq, wq = _codes(M, K, 2100), _codes(N, K, 2200)
    g = torch.Generator().manual_seed(2300)
    sx = (torch.rand(M, generator=g) * 1e-3 + 1e-4).to(dev)
    sw = (torch.rand(N, generator=g) * 1e-3 + 1e-4).to(dev)
    xq16, w16 = xq.to(torch.float16).to(dev), wq.to(torch.float16).to(dev)
    y_auto = ck.int8_gemm_dequant(xq16, sx, w16, sw)
    ck.debug_force_gemm_tile(2128)
    try:
        y_pairs = ck.int8_gemm_dequant(xq16, sx, w16, sw)
        poll_ok()
    finally:
        ck.debug_force_gemm_tile(0)
    assert torch.equal(y_auto, y_pairs)


def test_split_k_residual_in_place():
    # the split-K epilogue with the residual being the output itself: each
    # 16-byte residual piece is read before the group's stores, so y = x W^T + y
    # equals the out-of-place result bit for bit
    dev = device()
    M, N, K = 300, 264, 8192
    xq, wq = _codes(M, K, 2400), _codes(N, K, 2500)
    g = torch.Generator().manual_seed(2600)
    sx = (torch.rand(M, generator=g) * 1e-3 + 1e-4).to(dev)
    sw = (torch.rand(N, generator=g) * 1e-3 + 1e-4).to(dev)
    b = (torch.randn(N, generator=g) * 0.5).to(torch.bfloat16).to(dev)
    r = (torch.randn(M, N, generator=g) * 2).to(torch.bfloat16).to(dev)
    xq16, w16 = xq.to(torch.float16).to(dev), wq.to(torch.float16).to(dev)
    ck.debug_force_gemm_tile(4512)
    try:
        y = ck.int8_gemm_dequant(xq16, sx, w16, sw, bias=b, residual=r)
        y_in = r.clone()
        ck.int8_gemm_dequant(xq16, sx, w16, sw, bias=b, residual=y_in, out=y_in)
        poll_ok()
    finally:
        ck.debug_force_gemm_tile(0)
    assert torch.equal(y, y_in)
    acc = torch.from_numpy(oracle.int8_gemm(xq.numpy(), wq.numpy()))
    y_ref = ((acc.double().float() * sx.cpu()[:, None] * sw.cpu()[None, :] + b.cpu().float()[None, :])
             + r.cpu().float()).to(torch.bfloat16)
    assert (y.cpu().float() - y_ref.float()).abs().max().item() <= 0.05 * y_ref.float().abs().max().item()
