"""Randomised parity sweep over the shapes the workloads do not visit: seeded
random (M, K, N, group, input act, bias, residual, weight layout) for the
linear, and (M, K, N, code width, bias, residual) for the small-M GEMV, each
against the oracle at the contract's tolerances; the GEMV's int32 sums also
bit for bit.  The draws are fixed by the seed, so a failure reproduces."""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_group_gb300 as ck
from swiglu_mlp_group_gb300 import workloads as wl

from gpu_helpers import assert_output_close, device, poll_ok

pytestmark = pytest.mark.gpu


def _draws(seed, n, fn):
    rng = np.random.default_rng(seed)
    return [fn(rng, i) for i in range(n)]


def _linear_case(rng, i):
    g = int(rng.choice([64, 128, 256]))
    K = g * int(rng.integers(1, 4096 // g + 1))
    return dict(M=int(rng.integers(1, 700)), K=K, N=8 * int(rng.integers(1, 160)), g=g,
                act=str(rng.choice(["none", "swiglu"])), bias=bool(rng.integers(0, 2)),
                residual=bool(rng.integers(0, 2)),
                layout=int(rng.choice([ck.CK_WLAYOUT_ROWMAJOR_I8, ck.CK_WLAYOUT_GEMM_F16])),
                seed=5000 + 11 * i)


def _long_k_case(rng, i):
    # few tiles, K >= 6144: the GEMM splits K between two CTA pairs
    g = int(rng.choice([64, 128, 256]))
    K = g * int(rng.integers(6144 // g, 12288 // g + 1))
    return dict(M=int(rng.integers(1, 129)), K=K, N=8 * int(rng.integers(1, 129)), g=g,
                act=str(rng.choice(["none", "swiglu"])), bias=bool(rng.integers(0, 2)),
                residual=bool(rng.integers(0, 2)),
                layout=int(rng.choice([ck.CK_WLAYOUT_ROWMAJOR_I8, ck.CK_WLAYOUT_GEMM_F16])),
                seed=7000 + 13 * i)


LINEAR_CASES = _draws(20260, 24, _linear_case) + _draws(20261, 6, _long_k_case)


@pytest.mark.parametrize("c", LINEAR_CASES, ids=lambda c: f"M{c['M']}K{c['K']}N{c['N']}g{c['g']}{c['act']}")
def test_linear_random_shape(c):
    dev = device()
    M, K, N, g, act = c["M"], c["K"], c["N"], c["g"], c["act"]
    Kin = 2 * K if act == "swiglu" else K
    x = wl.activation(M, Kin, c["seed"], 0.01, 20.0)
    W = wl.weight(N, K, c["seed"] + 1)
    b = wl.bias(N, c["seed"] + 2) if c["bias"] else None
    r = wl.activation(M, N, c["seed"] + 3) if c["residual"] else None
    Wq, sw = ck.quantize_weight(W.to(dev), g)
    Wd = Wq if c["layout"] == ck.CK_WLAYOUT_ROWMAJOR_I8 else ck.prepare_weight(Wq, sw, c["layout"])
    y = ck.int8_linear(x.to(dev), Wd, sw, g, bias=None if b is None else b.to(dev), act=act,
                       wlayout=c["layout"], N=N, residual=None if r is None else r.to(dev))
    poll_ok()
    Wq_o, sw_o = oracle.quantize_weight(W.numpy(), g)
    y_o = oracle.int8_linear(wl.bf16_bits(x), Wq_o, sw_o, g, None if b is None else wl.bf16_bits(b),
                             act, residual_bits=None if r is None else wl.bf16_bits(r))
    assert_output_close(y, y_o)


def _gemv_case(rng, i):
    g = int(rng.choice([64, 128, 256]))
    K = g * int(rng.integers(1, 8192 // g + 1))
    return dict(M=int(rng.integers(1, 9)), K=K, N=8 * int(rng.integers(1, 400)), g=g,
                bits=int(rng.choice([8, 6, 4])), bias=bool(rng.integers(0, 2)),
                residual=bool(rng.integers(0, 2)), seed=6000 + 13 * i)


GEMV_CASES = _draws(20261, 24, _gemv_case)


@pytest.mark.parametrize("c", GEMV_CASES, ids=lambda c: f"M{c['M']}K{c['K']}N{c['N']}W{c['bits']}")
def test_gemv_random_shape(c):
    dev = device()
    M, K, N, g, bits = c["M"], c["K"], c["N"], c["g"], c["bits"]
    layout = ck.GEMV_LAYOUT_OF_BITS[bits]
    x = wl.activation(M, K, c["seed"], 0.01, 20.0)
    W = wl.weight(N, K, c["seed"] + 1)
    b = wl.bias(N, c["seed"] + 2) if c["bias"] else None
    r = wl.activation(M, N, c["seed"] + 3) if c["residual"] else None
    Wq, sw = ck.quantize_weight_bits(W.to(dev), g, bits)
    Wp = ck.prepare_weight(Wq, sw, layout)
    y = ck.gemv_smallM(x.to(dev), Wp, N, g, bias=None if b is None else b.to(dev),
                       residual=None if r is None else r.to(dev), wlayout=layout)
    xq, _ = ck.rotate_quantize_act(x.to(dev), g)
    acc = ck.debug_gemv_s32(xq, Wp, layout, N)
    poll_ok()
    Wq_o, sw_o = oracle.quantize_weight_bits(W.numpy(), g, bits)
    y_o = oracle.int8_linear(wl.bf16_bits(x), Wq_o, sw_o, g, None if b is None else wl.bf16_bits(b),
                             residual_bits=None if r is None else wl.bf16_bits(r))
    assert_output_close(y, y_o)
    # the sums on the GPU's own codes (both sides integer: exact)
    want = oracle.int8_gemm(xq.cpu().numpy(), Wq.cpu().numpy()) * (1 << (8 - bits))
    np.testing.assert_array_equal(acc.cpu().numpy().astype(np.int64), want)
