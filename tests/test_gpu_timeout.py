"""Failure detection without a GPU fault: a kernel whose pipeline barrier is
never completed gives up after the configured time limit, records
CK_ERR_TIMEOUT in the device status word and returns; the context stays usable
and the status word is cleared once read."""
import pytest
import torch

import oracle
import swiglu_mlp_group_gb300 as ck
from swiglu_mlp_group_gb300 import workloads as wl

from gpu_helpers import assert_output_close, device

pytestmark = pytest.mark.gpu


def test_stalled_wait_reports_timeout_and_context_survives():
    dev = device()
    assert ck.poll_device_status() == ck.CK_OK
    ck.set_wait_timeout_ns(50_000_000)  # 50 ms
    try:
        assert ck.debug_stalled_wait() == ck.CK_OK
        assert ck.poll_device_status() == ck.CK_ERR_TIMEOUT
        assert ck.poll_device_status() == ck.CK_OK  # cleared on read
    finally:
        ck.set_wait_timeout_ns(0)
    # the context still works
    c = wl.LINEAR_TINY
    x, W = c.x(), c.W()
    Wq, sw = ck.quantize_weight(W.to(dev), c.g)
    y = ck.int8_linear(x.to(dev), Wq, sw, c.g)
    Wq_o, sw_o = oracle.quantize_weight(W.numpy(), c.g)
    assert_output_close(y, oracle.int8_linear(wl.bf16_bits(x), Wq_o, sw_o, c.g))
    assert ck.poll_device_status() == ck.CK_OK
