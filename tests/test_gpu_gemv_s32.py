"""The small-M GEMV's exact int32 sums against the oracle's int64 GEMM, bit
for bit (ck_debug_gemv_s32: the engines' sums before the dequantization): all
three weight code widths on the INT8 grid (the 6- / 4-bit codes times 4 / 16),
every engine (dp4a for 1-4 tokens, the INT8 MMA beyond), activation
fragments staged in shared memory and read through L1, ragged tiles, and
adversarial all-maximum sign patterns at the largest sums."""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_group_gb300 as ck

from gpu_helpers import device, poll_ok

pytestmark = pytest.mark.gpu

LAYOUT = {8: ck.CK_WLAYOUT_GEMV_PACKED, 6: ck.CK_WLAYOUT_GEMV_PACKED_W6,
          4: ck.CK_WLAYOUT_GEMV_PACKED_W4}


def _check(xq, Wq, bits):
    dev = device()
    N = Wq.shape[0]
    Wp = ck.prepare_weight(torch.as_tensor(Wq).to(dev), torch.ones(N, device=dev), LAYOUT[bits])
    acc = ck.debug_gemv_s32(torch.as_tensor(xq).to(dev), Wp, LAYOUT[bits], N)
    poll_ok()
    want = oracle.int8_gemm(xq, Wq) * (1 << (8 - bits))
    np.testing.assert_array_equal(acc.cpu().numpy().astype(np.int64), want)


@pytest.mark.parametrize("bits", [8, 6, 4])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("N,K", [(40, 256), (1032, 4096), (264, 16384)])
def test_gemv_sums_exact(bits, M, N, K):
    rng = np.random.default_rng(4000 + 7 * M + K + bits)
    qmax = (1 << (bits - 1)) - 1
    xq = rng.integers(-127, 128, size=(M, K), dtype=np.int64).astype(np.int8)
    Wq = rng.integers(-qmax, qmax + 1, size=(N, K), dtype=np.int64).astype(np.int8)
    _check(xq, Wq, bits)


@pytest.mark.parametrize("bits", [8, 6, 4])
@pytest.mark.parametrize("M", [2, 8])
def test_gemv_sums_extreme_at_k_12288(bits, M):
    # |sum| up to 12288 * 127 * 127 (INT8) / 127 * 112 (4-bit on the grid): the
    # largest sums any workload reaches, both signs, in every row and token
    K, N = 12288, 48
    qmax = (1 << (bits - 1)) - 1
    xq = np.full((M, K), 127, np.int8)
    xq[1::2] = -127
    Wq = np.full((N, K), qmax, np.int8)
    Wq[1::3] = -qmax
    Wq[2::3, ::2] = -qmax  # half the products negative: sum 0
    _check(xq, Wq, bits)
