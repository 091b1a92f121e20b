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
