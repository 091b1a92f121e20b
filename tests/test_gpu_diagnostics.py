"""The two tensor-core rate diagnostics the measurements quote peaks against
return plausible numbers for a GB300 and leave the device status clean: the
legacy INT8 mma.sync rate (the only INT8 tensor instruction sm_103a has) and
the issue rate of the tcgen05 kind::f16 instruction the GEMMs run on."""
import pytest

import swiglu_mlp_group_gb300 as ck

from gpu_helpers import device, poll_ok

pytestmark = pytest.mark.gpu


def test_int8_mma_sync_rate():
    device()
    tops = ck.measure_int8_mma_tops()
    assert 20.0 < tops < 2000.0, tops
    poll_ok()


def test_tcgen05_f16_issue_rate():
    device()
    tflops = ck.measure_tcgen05_f16_tflops()
    # 128 SM cycles per 128x256x16 instruction at 1-2.1 GHz on 152 SMs: ~1.2-2.6 PFLOP/s
    assert 1000.0 < tflops < 3000.0, tflops
    poll_ok()


@pytest.mark.parametrize("pair", [False, True])
@pytest.mark.parametrize("n", [64, 128, 224, 256])
def test_tcgen05_rate_by_shape(n, pair):
    device()
    tflops, ns = ck.debug_tcgen05_rate(n, pair)
    assert 500.0 < tflops < 3000.0, (n, pair, tflops)
    # at least the tensor core's flops: 2 x 128 x n x 16 per SM at <= ~2.1 GHz x 8192 flop/clk
    assert ns > 1e9 * 2 * 128 * n * 16 / (8192 * 2.1e9) * 0.9, (n, pair, ns)
    poll_ok()


def test_tcgen05_rate_rejects_other_widths():
    assert ck.lib().ck_debug_tcgen05_rate(96, 0, None, None, None) == ck.CK_ERR_NULL


def test_streaming_read_bandwidth():
    device()
    small = ck.debug_read_bandwidth(50 << 20)
    large = ck.debug_read_bandwidth(800 << 20, nslices=2)
    assert 1000.0 < small < 12000.0 and 1000.0 < large < 12000.0, (small, large)
    poll_ok()


@pytest.mark.parametrize("n", [128, 224, 256])
def test_mma_issue_loop_forms(n):
    # every form ends with a clean status; with the MMAs' own time as the floor
    # (n / 2 SM cycles per instruction, four per k-block, at most ~2.1 GHz), the
    # GEMMs' loop form costs no more per k-block than the one it replaced
    device()
    ns = [ck.debug_mma_issue_loop(n, form) for form in (0, 1, 2)]
    poll_ok()
    floor_ns = 4 * (n / 2) / 2.1
    assert all(floor_ns * 0.95 < v < 10000.0 for v in ns), ns
    assert ns[2] <= ns[1] * 1.02, ns


def test_mma_issue_loop_rejects_other_arguments():
    device()
    for n, form in [(64, 0), (128, 3), (256, -1)]:
        with pytest.raises(ck.CkError):
            ck.debug_mma_issue_loop(n, form)
