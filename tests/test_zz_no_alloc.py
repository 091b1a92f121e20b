"""ck_int8_linear_noalloc: the ConvRot linear for callers that cannot allocate
device memory (hosts that own and pre-plan all device memory, such as an
inference engine's plugin step, or C callers without an allocator).  Its
temporaries live in the library's built-in device scratch array instead of a
caller workspace.

Checked through the C ABI against ck_int8_linear (the workspace entry point)
within the output tolerance of the other tests, on two calls in a row with
different shapes and inputs, so a stale scratch from the first call would
show in the second.  This file is collected last; it also passes alone in a
fresh process, where its first call sets up the scratch address.
"""
import pytest
import torch

import oracle
import swiglu_mlp_group_gb300 as ck
from swiglu_mlp_group_gb300 import workloads as wl

from gpu_helpers import OUT_REL_L2, device, poll_ok

pytestmark = pytest.mark.gpu


def _noalloc(x, W16, sw, g, bias, N, act=ck.CK_ACT_NONE, K=None):
    M, ldx = x.shape
    K = K if K is not None else (ldx // 2 if act == ck.CK_ACT_SWIGLU else ldx)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    st = ck.ck_int8_linear_noalloc(x.data_ptr(), M, K, ldx, act, W16.data_ptr(), sw.data_ptr(),
                                   N, g, None if bias is None else bias.data_ptr(), None,
                                   y.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == ck.CK_OK, ck.status_string(st)
    return y


def test_noalloc_matches_workspace_entry_point_two_calls_in_a_row():
    dev = device()
    cases = [(wl.LINEAR_2048, None), (wl.LINEAR_TINY, wl.LINEAR_TINY.b())]
    for c, b in cases:
        x = c.x().to(dev)
        Wq, sw = ck.quantize_weight(c.W().to(dev), c.g)
        W16 = ck.prepare_weight(Wq, sw, ck.CK_WLAYOUT_GEMM_F16)
        bias = None if b is None else b.to(dev)
        y_ref = ck.int8_linear(x, W16, sw, c.g, bias=bias, wlayout=ck.CK_WLAYOUT_GEMM_F16)
        y = _noalloc(x, W16, sw, c.g, bias, c.N)
        torch.cuda.synchronize()
        err = oracle.rel_l2(y.float().cpu().numpy(), y_ref.float().cpu().numpy())
        assert err <= OUT_REL_L2, (c.name, err)
    poll_ok()


def test_noalloc_swiglu_act_and_size_limit():
    dev = device()
    M, I, N, g = 64, 512, 256, 128
    h = wl.activation(M, 2 * I, seed=51).to(dev)
    Wq, sw = ck.quantize_weight(wl.weight(N, I, seed=52).to(dev), g)
    W16 = ck.prepare_weight(Wq, sw, ck.CK_WLAYOUT_GEMM_F16)
    y_ref = ck.int8_linear(h, W16, sw, g, act="swiglu", wlayout=ck.CK_WLAYOUT_GEMM_F16)
    y = _noalloc(h, W16, sw, g, None, N, act=ck.CK_ACT_SWIGLU)
    torch.cuda.synchronize()
    assert oracle.rel_l2(y.float().cpu().numpy(), y_ref.float().cpu().numpy()) <= OUT_REL_L2
    # beyond the built-in scratch: rejected before anything is launched
    big_M, big_K = 8192, 4096
    assert big_M * big_K * 2 > 32 * 1024 * 1024
    st = ck.ck_int8_linear_noalloc(h.data_ptr(), big_M, big_K, big_K, ck.CK_ACT_NONE,
                                   W16.data_ptr(), sw.data_ptr(), N, g, None, None, y.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    assert st == ck.CK_ERR_WORKSPACE
    poll_ok()


def test_noalloc_chain_with_overlapped_launches():
    # every call reuses the one scratch array: the next call's quantizer must
    # wait for the previous GEMM before it overwrites the codes it reads
    dev = device()
    M, K, g = 512, 1024, 128
    layers = []
    for i in range(4):
        Wq, sw = ck.quantize_weight(wl.weight(K, K, 1200 + i).to(dev), g)
        layers.append((ck.prepare_weight(Wq, sw, ck.CK_WLAYOUT_GEMM_F16), sw))
    torch.cuda.synchronize()
    x0 = wl.activation(M, K, 1210).to(dev)

    def chain(sync_each):
        x, outs = x0, []
        for W16, sw in layers:
            x = _noalloc(x, W16, sw, g, None, K)
            if sync_each:
                torch.cuda.synchronize()
            outs.append(x)
        torch.cuda.synchronize()
        return outs

    ref = chain(True)
    ck.set_launch_overlap(True)
    try:
        got = chain(False)
    finally:
        ck.set_launch_overlap(False)
    for a, b in zip(got, ref):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    poll_ok()
