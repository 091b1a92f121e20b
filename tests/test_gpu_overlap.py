"""Overlapped launches (ck_set_launch_overlap) change when kernels start, never
what they compute.  Chains of calls in which every call reads the previous
call's output and reuses one workspace give bit-identical results with the mode
on and off, eagerly and replayed from a CUDA graph.  A kernel that read its
activation operand, or overwrote a shared workspace, before the kernel ahead of
it had finished would show up here as a mismatch."""
import pytest
import torch

import swiglu_mlp_group_gb300 as ck
from swiglu_mlp_group_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
G = 128


def _bits(t):
    return t.view(torch.int16)


def _weights(n_layers, N, K, layout, seed):
    out = []
    for i in range(n_layers):
        Wq, sw = ck.quantize_weight(wl.weight(N, K, seed + i).to(DEV), G)
        out.append((ck.prepare_weight(Wq, sw, layout) if layout != ck.CK_WLAYOUT_ROWMAJOR_I8 else Wq,
                    sw))
    torch.cuda.synchronize()  # settled before any overlapped use
    return out


def _run(chain, overlap, sync_each):
    ck.set_launch_overlap(overlap)
    try:
        outs = chain(sync_each)
        torch.cuda.synchronize()
        assert ck.poll_device_status() == ck.CK_OK
        return [o.clone() for o in outs]
    finally:
        ck.set_launch_overlap(False)


def _check_chain(chain):
    ref = _run(chain, False, True)
    for overlap in (False, True):
        got = _run(chain, overlap, False)
        assert len(got) == len(ref)
        for i, (a, b) in enumerate(zip(got, ref)):
            assert torch.equal(_bits(a), _bits(b)), f"layer {i} differs (overlap={overlap})"


@pytest.mark.parametrize("M,K,layout", [(256, 1024, ck.CK_WLAYOUT_GEMM_F16),
                                        (2048, 4096, ck.CK_WLAYOUT_GEMM_F16),
                                        (256, 1024, ck.CK_WLAYOUT_ROWMAJOR_I8)])
def test_linear_chain(M, K, layout):
    layers = _weights(5, K, K, layout, 100)
    x0 = wl.activation(M, K, 7).to(DEV)
    bias = (torch.randn(K, generator=torch.Generator().manual_seed(3)) * 0.02).to(torch.bfloat16).to(DEV)
    ws = torch.empty(ck.workspace_bytes(ck.CK_OP_INT8_LINEAR, M, K, K, layout), dtype=torch.uint8,
                     device=DEV)
    ys = [torch.empty(M, K, dtype=torch.bfloat16, device=DEV) for _ in layers]

    def chain(sync_each):
        x = x0
        for i, (W, sw) in enumerate(layers):
            # odd layers add their input back (residual = the layer's own input)
            ck.int8_linear(x, W, sw, G, bias=bias, wlayout=layout, out=ys[i], workspace=ws,
                           residual=x if i % 2 else None)
            if sync_each:
                torch.cuda.synchronize()
            x = ys[i]
        return ys

    _check_chain(chain)


@pytest.mark.parametrize("layout", [ck.CK_WLAYOUT_GEMM_F16, ck.CK_WLAYOUT_ROWMAJOR_I8])
def test_mlp_chain(layout):
    # with INT8 row-major weights each call widens gate|up, then down, into the
    # same workspace slot: the second widening must wait for the first GEMM
    M, H, I = 512, 1024, 1536
    gus = _weights(3, 2 * I, H, layout, 200)
    downs = _weights(3, H, I, layout, 300)
    x0 = wl.activation(M, H, 8).to(DEV)
    ws = torch.empty(ck.workspace_bytes(ck.CK_OP_SWIGLU_MLP, M, H, I, layout),
                     dtype=torch.uint8, device=DEV)
    ys = [torch.empty(M, H, dtype=torch.bfloat16, device=DEV) for _ in gus]

    def chain(sync_each):
        x = x0
        for i in range(len(gus)):
            ck.swiglu_mlp(x, gus[i][0], gus[i][1], downs[i][0], downs[i][1], G,
                          wlayout=layout, out=ys[i], workspace=ws, residual=x)
            if sync_each:
                torch.cuda.synchronize()
            x = ys[i]
        return ys

    _check_chain(chain)


@pytest.mark.parametrize("M", [1, 2, 5, 8])
def test_gemv_chain(M):
    K = 4096
    layers = _weights(6, K, K, ck.CK_WLAYOUT_GEMV_PACKED, 400)
    x0 = wl.activation(M, K, 9).to(DEV)
    ws = torch.empty(ck.workspace_bytes(ck.CK_OP_GEMV_SMALLM, M, K, K), dtype=torch.uint8,
                     device=DEV)
    ys = [torch.empty(M, K, dtype=torch.bfloat16, device=DEV) for _ in layers]

    def chain(sync_each):
        x = x0
        for i, (Wp, _) in enumerate(layers):
            if i % 3 == 2:
                # the standalone pair: quantizer call, then the GEMV on its codes
                xq, sx = ck.rotate_quantize_act(x, G)
                ck.int8_gemv_dequant(xq, sx, Wp, K, out=ys[i], residual=x)
            else:
                ck.gemv_smallM(x, Wp, K, G, out=ys[i], workspace=ws)
            if sync_each:
                torch.cuda.synchronize()
            x = ys[i]
        return ys

    _check_chain(chain)


def test_graph_replay_of_an_overlapped_chain():
    M, K = 4, 4096
    lin = _weights(2, K, K, ck.CK_WLAYOUT_GEMM_F16, 500)
    gv = _weights(2, K, K, ck.CK_WLAYOUT_GEMV_PACKED, 600)
    x0 = wl.activation(M, K, 10).to(DEV)
    ws_l = torch.empty(ck.workspace_bytes(ck.CK_OP_INT8_LINEAR, M, K, K, ck.CK_WLAYOUT_GEMM_F16),
                       dtype=torch.uint8, device=DEV)
    ws_g = torch.empty(ck.workspace_bytes(ck.CK_OP_GEMV_SMALLM, M, K, K), dtype=torch.uint8,
                       device=DEV)
    ys = [torch.empty(M, K, dtype=torch.bfloat16, device=DEV) for _ in range(4)]

    def chain(stream):
        x = x0
        for i in range(4):
            if i % 2 == 0:
                W, sw = lin[i // 2]
                ck.int8_linear(x, W, sw, G, wlayout=ck.CK_WLAYOUT_GEMM_F16, out=ys[i],
                               workspace=ws_l, stream=stream)
            else:
                ck.gemv_smallM(x, gv[i // 2][0], K, G, out=ys[i], workspace=ws_g, stream=stream)
            x = ys[i]

    ck.set_launch_overlap(False)
    chain(None)
    torch.cuda.synchronize()
    ref = [y.clone() for y in ys]
    for y in ys:
        y.fill_(0)
    ck.set_launch_overlap(True)
    try:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            chain(s)  # warm-up outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            chain(s)
        for _ in range(3):
            for y in ys:
                y.fill_(0)
            g.replay()
            torch.cuda.synchronize()
            for a, b in zip(ys, ref):
                assert torch.equal(_bits(a), _bits(b))
    finally:
        ck.set_launch_overlap(False)
    assert ck.poll_device_status() == ck.CK_OK
