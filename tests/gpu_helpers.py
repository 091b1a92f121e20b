"""Shared helpers of the GPU parity tests (tolerances of the contract)."""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_group_gb300 as ck

# INT8 codes may differ by +-1 at rounding ties on at most this fraction
CODE_MISMATCH_FRACTION = 1e-4
# weight codes: the offline weight rotation runs in float64 like the oracle's,
# so only a float64 rounding coincidence can flip a code
WEIGHT_CODE_MISMATCH_FRACTION = 1e-6
# per-row scales: f32 butterflies vs the oracle's float64 rotation
SCALE_RTOL = 1e-6
# bf16 outputs: relative L2 against the oracle
OUT_REL_L2 = 2e-3


def device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    ck.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    assert ck.ck_device_check() == ck.CK_OK, "not a compute capability 10.3 device"
    return d


def assert_codes_match(q_gpu, q_ref, what="codes", fraction=CODE_MISMATCH_FRACTION):
    q_gpu = np.asarray(q_gpu, dtype=np.int32)
    q_ref = np.asarray(q_ref, dtype=np.int32)
    assert q_gpu.shape == q_ref.shape
    d = np.abs(q_gpu - q_ref)
    assert d.max(initial=0) <= 1, f"{what}: a code differs by {d.max()}"
    n_bad = int(np.count_nonzero(d))
    assert n_bad <= fraction * d.size, (
        f"{what}: {n_bad} of {d.size} codes differ by 1 (> {fraction:g})")


def assert_scales_match(s_gpu, s_ref, what="scales"):
    s_gpu = np.asarray(s_gpu, np.float64)
    s_ref = np.asarray(s_ref, np.float64)
    np.testing.assert_allclose(s_gpu, s_ref, rtol=SCALE_RTOL, atol=0, err_msg=what)


def bf16_to_np(t):
    return t.float().cpu().numpy()


def assert_output_close(y_gpu, y_ref_bits, what="y"):
    err = oracle.rel_l2(bf16_to_np(y_gpu), oracle.bf16_bits_to_f32(y_ref_bits))
    assert err <= OUT_REL_L2, f"{what}: rel L2 {err:.3e} > {OUT_REL_L2}"
    return err


def poll_ok():
    assert ck.poll_device_status() == ck.CK_OK
