"""ck_int8_linear_noalloc: the ConvRot linear for callers that cannot allocate
device memory (hosts that own and pre-plan all device memory, such as an
inference engine's plugin step, or C callers without an allocator).  Its
temporaries live in the library's built-in device scratch array instead of a
caller workspace.

Both entry points run the same kernels on the same arithmetic, so the checks
here are bit-for-bit against ck_int8_linear (the workspace entry point) on
the GEMM-resident weight layout, with bias, residual and an in-place residual,
plus the oracle at the output tolerance of the other tests.  The size limit
is tested at its exact boundary.  Calls in a row share the scratch: a large call fills
it first, then a smaller one must overwrite every byte it reads; the
workspace of the reference call is filled with a different pattern, so codes
or scales left over from the large call would show as a mismatch.  This file
is collected last; it also passes alone in a fresh process, where its first
call sets up the scratch address.
"""
import pytest
import torch

import oracle
import swiglu_mlp_group_gb300 as ck
from swiglu_mlp_group_gb300 import workloads as wl

from gpu_helpers import assert_output_close, device, poll_ok

pytestmark = pytest.mark.gpu

SCRATCH = 32 * 1024 * 1024  # CK_NOALLOC_SCRATCH_BYTES


LAY = ck.CK_WLAYOUT_GEMM_F16  # the layout the entry point takes


def _need(M, K):
    """Scratch bytes of one call: fp16-held codes (rounded to 256 bytes), then f32 scales."""
    return (2 * M * K + 255) // 256 * 256 + 4 * M


def _noalloc(x, W, sw, g, N, wlayout=LAY, bias=None, residual=None, out=None,
             act=ck.CK_ACT_NONE):
    assert wlayout == LAY
    M, ldx = x.shape
    K = ldx // 2 if act == ck.CK_ACT_SWIGLU else ldx
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    st = ck.ck_int8_linear_noalloc(x.data_ptr(), M, K, ldx, act, W.data_ptr(), sw.data_ptr(), N, g,
                                   None if bias is None else bias.data_ptr(),
                                   None if residual is None else residual.data_ptr(),
                                   y.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == ck.CK_OK, ck.status_string(st)
    return y


def _reference(x, W, sw, g, N, wlayout, bias=None, residual=None, act="none"):
    """ck_int8_linear with a workspace filled with 0x55 bytes (not the noalloc
    scratch's leftovers)."""
    M, ldx = x.shape
    K = ldx // 2 if act == "swiglu" else ldx
    ws = torch.full((ck.workspace_bytes(ck.CK_OP_INT8_LINEAR, M, K, N, wlayout),), 0x55,
                    dtype=torch.uint8, device=x.device)
    return ck.int8_linear(x, W, sw, g, bias=bias, act=act, N=N, wlayout=wlayout, workspace=ws,
                          residual=residual)


def _weights(N, K, g, seed, wlayout, dev):
    Wq, sw = ck.quantize_weight(wl.weight(N, K, seed).to(dev), g)
    W = Wq if wlayout == ck.CK_WLAYOUT_ROWMAJOR_I8 else ck.prepare_weight(Wq, sw, wlayout)
    return Wq, W, sw


def test_noalloc_equals_workspace_entry_point_and_oracle_two_calls_in_a_row():
    dev = device()
    wlayout = LAY
    # call 1: a large linear that fills most of the scratch
    big = wl.LINEAR_2048
    xb = big.x().to(dev)
    _, Wb, swb = _weights(big.N, big.K, big.g, 1000 * big.seed + 2, wlayout, dev)
    y1 = _noalloc(xb, Wb, swb, big.g, big.N, wlayout)
    assert torch.equal(y1, _reference(xb, Wb, swb, big.g, big.N, wlayout))
    # call 2: the tiny linear with bias, reading the start of the same scratch
    c = wl.LINEAR_TINY
    x, b = c.x().to(dev), c.b().to(dev)
    Wq, W, sw = _weights(c.N, c.K, c.g, 1000 * c.seed + 2, wlayout, dev)
    y2 = _noalloc(x, W, sw, c.g, c.N, wlayout, bias=b)
    y_ref = _reference(x, W, sw, c.g, c.N, wlayout, bias=b)
    poll_ok()
    assert torch.equal(y2, y_ref)
    y_o = oracle.int8_linear(wl.bf16_bits(c.x()), Wq.cpu().numpy(), sw.cpu().numpy(), c.g,
                             wl.bf16_bits(c.b()))
    assert_output_close(y2, y_o)


def test_noalloc_residual_and_in_place_residual():
    dev = device()
    M, K, N, g = 300, 1024, 520, 128
    x = wl.activation(M, K, 1101, 0.005, 30.0).to(dev)
    b = wl.bias(N, 1102).to(dev)
    r = (torch.randn(M, N, generator=torch.Generator().manual_seed(1103)) * 4).to(torch.bfloat16)
    r = r.to(dev)
    Wq, W, sw = _weights(N, K, g, 1104, LAY, dev)
    lay = LAY
    y_ref = _reference(x, W, sw, g, N, lay, bias=b, residual=r)
    y = _noalloc(x, W, sw, g, N, lay, bias=b, residual=r)
    y_in = r.clone()
    _noalloc(x, W, sw, g, N, lay, bias=b, residual=y_in, out=y_in)  # residual is y
    poll_ok()
    assert torch.equal(y, y_ref)
    assert torch.equal(y_in, y_ref)


def test_noalloc_swiglu_input_activation():
    dev = device()
    M, I, N, g = 64, 512, 256, 128
    h = wl.activation(M, 2 * I, seed=51).to(dev)
    _, W, sw = _weights(N, I, g, 52, LAY, dev)
    lay = LAY
    y = _noalloc(h, W, sw, g, N, lay, act=ck.CK_ACT_SWIGLU)
    poll_ok()
    assert torch.equal(y, _reference(h, W, sw, g, N, lay, act="swiglu"))


def test_noalloc_size_limit_exact_boundary():
    # K = 4096: 4094 rows fill the scratch to within 8 bytes (the scales end at
    # its last bytes) and are accepted; 4095 rows are rejected before launch
    dev = device()
    K, N, g = 4096, 256, 128
    M_max = 4094
    assert _need(M_max, K) <= SCRATCH < _need(M_max + 1, K)
    assert SCRATCH - _need(M_max, K) == 8
    x = wl.activation(M_max + 1, K, 1201, 0.005, 30.0).to(dev)
    _, W, sw = _weights(N, K, g, 1202, LAY, dev)
    lay = LAY
    xm = x[:M_max]
    y = _noalloc(xm, W, sw, g, N, lay)
    poll_ok()
    assert torch.equal(y, _reference(xm, W, sw, g, N, lay))
    y1 = torch.empty((M_max + 1, N), dtype=torch.bfloat16, device=dev)
    st = ck.ck_int8_linear_noalloc(x.data_ptr(), M_max + 1, K, K, ck.CK_ACT_NONE, W.data_ptr(),
                                   sw.data_ptr(), N, g, None, None, y1.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    assert st == ck.CK_ERR_WORKSPACE
    poll_ok()


def test_noalloc_chain_with_overlapped_launches():
    # every call reuses the one scratch array: the next call's quantizer must
    # wait for the previous GEMM before it overwrites the codes it reads
    dev = device()
    M, K, g = 512, 1024, 128
    lay = LAY
    layers = [_weights(K, K, g, 1200 + i, lay, dev)[1:] for i in range(4)]
    torch.cuda.synchronize()
    x0 = wl.activation(M, K, 1210).to(dev)

    def chain(sync_each):
        x, outs = x0, []
        for W, sw in layers:
            x = _noalloc(x, W, sw, g, K, lay)
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
        assert torch.equal(a, b)
    poll_ok()
