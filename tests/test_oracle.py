"""Pins for the CPU oracle: each check ties an oracle function to something other
than itself -- hand-worked fixtures under tests/golden/, closed forms, textbook
special cases, library routines and brute force on tiny inputs.  A plausible
mistake (dropped term, wrong sign or index, transposed operand, wrong rounding
mode) fails at least one of them.  CPU only.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from swiglu_mlp_group_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_hadamard_fixture():
    mats, g, rows = {}, None, []
    for line in open(os.path.join(GOLDEN, "hadamard_sylvester.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("g "):
            if g is not None:
                mats[g] = np.array(rows, dtype=np.float64)
            g, rows = int(line.split()[1]), []
        else:
            rows.append([float(t) for t in line.split()])
    mats[g] = np.array(rows, dtype=np.float64)
    return mats


# --------------------------------------------------------------------------
# Hadamard
# --------------------------------------------------------------------------

def test_hadamard_matches_hand_written_sylvester_fixture():
    for g, Hu in _read_hadamard_fixture().items():
        np.testing.assert_array_equal(oracle.hadamard(g) * math.sqrt(g), Hu)


@pytest.mark.parametrize("g", [1, 2, 4, 8, 16, 32, 64, 128, 256])
def test_hadamard_orthogonal_symmetric_and_pm_inv_sqrt_g(g):
    H = oracle.hadamard(g)
    assert np.max(np.abs(H - H.T)) == 0.0
    assert np.max(np.abs(H @ H.T - np.eye(g))) < 1e-14
    np.testing.assert_array_equal(np.abs(H), np.full((g, g), 1.0 / math.sqrt(g)))


@pytest.mark.parametrize("g", [2, 16, 64, 128, 256])
def test_hadamard_natural_order_closed_form_and_scipy(g):
    # Sylvester order has the closed form H[i, j] = (-1)^popcount(i & j).
    i = np.arange(g)[:, None]
    j = np.arange(g)[None, :]
    signs = np.vectorize(lambda a: (-1.0) ** bin(int(a)).count("1"))(i & j)
    np.testing.assert_array_equal(oracle.hadamard(g) * math.sqrt(g), signs)
    scipy_linalg = pytest.importorskip("scipy.linalg")
    np.testing.assert_array_equal(oracle.hadamard(g) * math.sqrt(g),
                                  scipy_linalg.hadamard(g).astype(np.float64))


def test_hadamard_rejects_non_power_of_two():
    with pytest.raises(ValueError):
        oracle.hadamard(96)


# --------------------------------------------------------------------------
# Rotation
# --------------------------------------------------------------------------

@pytest.mark.parametrize("g", [64, 128, 256])
def test_rotation_is_block_diagonal_over_contiguous_groups(g):
    K = 4 * g
    H = oracle.hadamard(g)
    # a unit vector inside group j rotates into row i of H_g, inside group j only
    for j, i in [(0, 0), (1, 5), (3, g - 1), (2, g // 2)]:
        e = np.zeros((1, K))
        e[0, j * g + i] = 1.0
        r = oracle.rotate_rows_f64(e, g)[0]
        expect = np.zeros(K)
        expect[j * g:(j + 1) * g] = H[i]
        np.testing.assert_array_equal(r, expect)


def test_rotation_identity_x_wt_equals_xrot_wrott():
    # comfy-kitchen PR #277, The key observation: x @ W^T == x_rot @ W_rot^T
    rng = np.random.default_rng(0)
    for g, K in [(64, 256), (128, 384), (256, 512)]:
        x = rng.standard_normal((5, K))
        W = rng.standard_normal((7, K))
        lhs = x @ W.T
        rhs = oracle.rotate_rows_f64(x, g) @ oracle.rotate_rows_f64(W, g).T
        assert np.max(np.abs(lhs - rhs)) <= 1e-12 * np.max(np.abs(lhs))


def test_rotation_preserves_row_norms():
    # sglang PR #35994 report, review notes: ConvRot keeps output-row L2 norms
    W = wl.weight(64, 512, seed=11).numpy()
    Wr = oracle.rotate_rows(W, 128)
    np.testing.assert_allclose(np.linalg.norm(Wr.astype(np.float64), axis=1),
                               np.linalg.norm(W.astype(np.float64), axis=1), rtol=1e-6)
    Wr64 = oracle.rotate_rows_f64(W.astype(np.float64), 128)
    np.testing.assert_allclose(np.linalg.norm(Wr64, axis=1),
                               np.linalg.norm(W.astype(np.float64), axis=1), rtol=1e-13)


def test_rotation_f32_is_f64_rounded_once():
    W = wl.weight(8, 256, seed=12).numpy()
    np.testing.assert_array_equal(oracle.rotate_rows(W, 64),
                                  oracle.rotate_rows_f64(W.astype(np.float64), 64)
                                  .astype(np.float32))


def test_rotation_rejects_ragged_groups():
    with pytest.raises(ValueError):
        oracle.rotate_rows(np.zeros((2, 200), np.float32), 64)


def test_rotation_group_one_is_identity():
    v = wl.weight(3, 40, seed=13).numpy()
    np.testing.assert_array_equal(oracle.rotate_rows(v, 1), v)


# --------------------------------------------------------------------------
# Quantizer
# --------------------------------------------------------------------------

def _read_quant_fixture():
    cases, cur = [], {}
    for line in open(os.path.join(GOLDEN, "quantize_rne_rows.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        cur[key] = [float(v) for v in vals]
        if key == "codes":
            cases.append(cur)
            cur = {}
    return cases


def test_quantizer_hand_worked_rows_ties_to_even():
    for case in _read_quant_fixture():
        v = np.array([case["row"]], dtype=np.float32)
        q, s = oracle.quantize_rows(v)
        np.testing.assert_array_equal(q[0], np.array(case["codes"], dtype=np.int8))
        assert s[0] == np.float32(case["scale"][0])


def test_quantizer_invariants_on_random_rows():
    v = wl.weight(200, 384, seed=14).numpy() * np.float32(3.0)
    v[7] = 0.0
    v[9] = -1.25
    q, s = oracle.quantize_rows(v)
    assert np.max(np.abs(q.astype(np.int32))) <= 127
    # the element of largest magnitude maps to +-127 (nonzero rows)
    for r in range(v.shape[0]):
        if r == 7:
            assert s[r] == 0.0 and not q[r].any()
            continue
        k = int(np.argmax(np.abs(v[r])))
        assert abs(int(q[r, k])) == 127
        assert np.sign(q[r, k]) == np.sign(v[r, k])
        assert s[r] == np.float32(np.max(np.abs(v[r]))) / np.float32(127.0)
    # reconstruction error at most half a step (f32 slack of a few ulp)
    err = np.abs(v.astype(np.float64) - q.astype(np.float64) * s[:, None].astype(np.float64))
    assert np.all(err <= s[:, None].astype(np.float64) * (0.5 + 1e-5))
    assert np.all(q[9] == -127)


def test_group_one_reduces_to_textbook_rowwise_w8a8():
    # g = 1 makes H the identity: plain per-row absmax INT8 quantization,
    # written here independently with numpy (np.rint rounds half to even).
    v = wl.weight(31, 64, seed=15).numpy() * np.float32(5.0)
    q, s = oracle.quantize_rows(oracle.rotate_rows(v, 1))
    s_ref = (np.max(np.abs(v), axis=1) / np.float32(127.0)).astype(np.float32)
    q_ref = np.clip(np.rint(v / s_ref[:, None]), -127, 127).astype(np.int8)
    np.testing.assert_array_equal(s, s_ref)
    np.testing.assert_array_equal(q, q_ref)


# --------------------------------------------------------------------------
# SwiGLU
# --------------------------------------------------------------------------

def test_swiglu_special_values_and_gate_up_order():
    h = np.array([[0.0, 1.0, 2.0, 40.0, -40.0,     # gates
                   5.0, 2.0, 1.0, 1.0, 1.0]],      # ups
                 dtype=np.float32)
    a = oracle.swiglu(h)[0].astype(np.float64)
    assert a[0] == 0.0                               # silu(0) = 0
    assert a[1] == np.float32(2.0 / (1.0 + math.exp(-1.0)))   # silu(1) * 2 (gate first)
    assert a[2] == np.float32(2.0 / (1.0 + math.exp(-2.0)))   # silu(2) * 1
    assert a[3] == np.float32(40.0)                  # silu(z) -> z for large z
    assert abs(a[4]) < 1e-15                         # silu(z) -> 0 for very negative z
    assert a[1] != a[2]


# --------------------------------------------------------------------------
# INT8 GEMM
# --------------------------------------------------------------------------

def test_gemm_brute_force_tiny_all_shapes():
    rng = np.random.default_rng(1)
    for M, N, K in [(1, 1, 1), (2, 3, 5), (3, 2, 7), (8, 8, 8), (5, 1, 6)]:
        xq = rng.integers(-127, 128, (M, K)).astype(np.int8)
        wq = rng.integers(-127, 128, (N, K)).astype(np.int8)
        acc = oracle.int8_gemm(xq, wq)
        for m in range(M):
            for n in range(N):
                s = 0
                for k in range(K):
                    s += int(xq[m, k]) * int(wq[n, k])
                assert acc[m, n] == s


def test_gemm_all_sign_patterns_k4():
    # every sign pattern of +-127 for K=4 on both operands
    pats = np.array([[127 if (b >> i) & 1 else -127 for i in range(4)] for b in range(16)],
                    dtype=np.int8)
    acc = oracle.int8_gemm(pats, pats)
    agree = np.array([[4 - 2 * bin(a ^ b).count("1") for b in range(16)] for a in range(16)])
    np.testing.assert_array_equal(acc, agree * 127 * 127)


def test_gemm_closed_forms_large_k():
    K = 12288
    ones = np.full((2, K), 127, dtype=np.int8)
    neg = np.full((3, K), -127, dtype=np.int8)
    np.testing.assert_array_equal(oracle.int8_gemm(ones, ones), np.full((2, 2), K * 16129))
    np.testing.assert_array_equal(oracle.int8_gemm(ones, neg), np.full((2, 3), -K * 16129))
    # float64 is exact for these integer sums (< 2^53): a library cross-check
    rng = np.random.default_rng(2)
    xq = rng.integers(-127, 128, (9, 1000)).astype(np.int8)
    wq = rng.integers(-127, 128, (11, 1000)).astype(np.int8)
    np.testing.assert_array_equal(oracle.int8_gemm(xq, wq),
                                  (xq.astype(np.float64) @ wq.astype(np.float64).T)
                                  .astype(np.int64))


# --------------------------------------------------------------------------
# bf16 rounding and dequantization
# --------------------------------------------------------------------------

def test_bf16_rounding_hand_worked_bit_patterns():
    for line in open(os.path.join(GOLDEN, "bf16_rne_bits.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        f_hex, b_hex = line.split()[:2]
        f = np.array([int(f_hex, 16)], dtype=np.uint32).view(np.float32)
        assert int(oracle.f32_to_bf16_bits(f)[0]) == int(b_hex, 16), line


def test_bf16_rounding_matches_torch_on_random_values():
    x = torch.randn(100000, generator=torch.Generator().manual_seed(3)) * 1e3
    x[:10] = torch.tensor([0.0, -0.0, 1e-40, -1e-40, 3.4e38, -3.4e38, 1.0, 2.0, 0.5, 7.0])
    ref = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.f32_to_bf16_bits(x.numpy()), ref)
    nan = oracle.f32_to_bf16_bits(np.array([np.nan], np.float32))
    assert oracle.bf16_bits_to_f32(nan)[0] != oracle.bf16_bits_to_f32(nan)[0]


def test_dequant_closed_form_and_bias_index():
    acc = np.array([[1, 2, 3], [4, 5, 6]], dtype=np.int64)
    sx = np.array([2.0, 0.5], dtype=np.float32)
    sw = np.array([3.0, 1.0, 0.25], dtype=np.float32)
    bias = oracle.f32_to_bf16_bits(np.array([0.5, -1.0, 2.0], np.float32))
    y = oracle.bf16_bits_to_f32(oracle.dequant(acc, sx, sw, bias))
    expect = np.array([[6.5, 3.0, 3.5], [6.5, 1.5, 2.75]], dtype=np.float32)
    np.testing.assert_array_equal(y, expect)
    y0 = oracle.bf16_bits_to_f32(oracle.dequant(acc, sx, sw, None))
    np.testing.assert_array_equal(y0, expect - np.array([0.5, -1.0, 2.0], np.float32))


def test_dequant_residual_closed_form_and_index():
    # [P2] Commits / Description: the residual joins the epilogue sum before the
    # single rounding; distinct values per (m, n) catch a transposed index
    acc = np.array([[1, 2, 3], [4, 5, 6]], dtype=np.int64)
    sx = np.array([2.0, 0.5], dtype=np.float32)
    sw = np.array([3.0, 1.0, 0.25], dtype=np.float32)
    bias = oracle.f32_to_bf16_bits(np.array([0.5, -1.0, 2.0], np.float32))
    res = oracle.f32_to_bf16_bits(np.array([[1.0, -2.0, 0.25], [0.125, 4.0, -8.0]], np.float32))
    y = oracle.bf16_bits_to_f32(oracle.dequant(acc, sx, sw, bias, res))
    expect = np.array([[7.5, 1.0, 3.75], [6.625, 5.5, -5.25]], dtype=np.float32)
    np.testing.assert_array_equal(y, expect)


def test_dequant_residual_matches_a_float64_sum_rounded_by_torch():
    rng = np.random.default_rng(7)
    M, N = 37, 53
    acc = rng.integers(-2 ** 24, 2 ** 24, size=(M, N)).astype(np.int64)
    sx = (rng.random(M) * 1e-3).astype(np.float32)
    sw = (rng.random(N) * 1e-2).astype(np.float32)
    b = torch.randn(N, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    r = (torch.randn(M, N, generator=torch.Generator().manual_seed(2)) * 30).to(torch.bfloat16)
    v = (torch.from_numpy(acc).double() * torch.from_numpy(sx).double()[:, None]
         * torch.from_numpy(sw).double()[None, :] + b.double()[None, :] + r.double())
    ref = v.to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.dequant(acc, sx, sw, b.view(torch.int16).numpy().view(np.uint16),
                         r.view(torch.int16).numpy().view(np.uint16))
    np.testing.assert_array_equal(got, ref)


def _tiny_linear_case():
    c = wl.LINEAR_TINY
    x = c.x()
    W = c.W().numpy()
    b = c.b()
    return c, x, W, b


def test_linear_error_bound_closed_form():
    """|y - y_ref| <= sum_k (|x_rot| sw/2 + |W_rot| sx/2 + 3 sx sw/4) + output rounding,
    from x_rot = sx*xq + ex, W_rot = sw*wq + ew with |ex| <= sx/2, |ew| <= sw/2."""
    c, x, W, b = _tiny_linear_case()
    xb = wl.bf16_bits(x)
    bb = wl.bf16_bits(b)
    Wq, sw = oracle.quantize_weight(W, c.g)
    y = oracle.bf16_bits_to_f32(oracle.int8_linear(xb, Wq, sw, c.g, bb)).astype(np.float64)
    xf = oracle.bf16_bits_to_f32(xb).astype(np.float64)
    y_ref = oracle.reference_linear_f64(xf, W, oracle.bf16_bits_to_f32(bb))
    xq, sx = oracle.rotate_quantize_act(xb, c.g)
    xr = np.abs(oracle.rotate_rows(oracle.bf16_bits_to_f32(xb), c.g).astype(np.float64))
    wr = np.abs(oracle.rotate_rows(W, c.g).astype(np.float64))
    sx64 = sx.astype(np.float64)[:, None]
    sw64 = sw.astype(np.float64)[None, :]
    bound = (xr.sum(1)[:, None] * sw64 / 2 + wr.sum(1)[None, :] * sx64 / 2
             + 0.75 * c.K * sx64 * sw64)
    bound += 1e-5 * (xr @ wr.T) + np.abs(y_ref) * 2.0 ** -8 + 1e-30
    assert np.all(np.abs(y - y_ref) <= bound)
    # INT8 noise level, the order of the pages' ~0.9% against float32
    assert 1e-3 < oracle.rel_l2(y, y_ref) < 3e-2


def test_linear_equals_composition_of_steps():
    c, x, W, b = _tiny_linear_case()
    xb = wl.bf16_bits(x)
    Wq, sw = oracle.quantize_weight(W, c.g)
    xq, sx = oracle.rotate_quantize_act(xb, c.g)
    y = oracle.int8_linear(xb, Wq, sw, c.g, None)
    np.testing.assert_array_equal(y, oracle.dequant(oracle.int8_gemm(xq, Wq), sx, sw, None))


# --------------------------------------------------------------------------
# SwiGLU MLP: fused vs staged (sglang PR #44196, Accuracy Tests)
# --------------------------------------------------------------------------

def _mlp_errors(M, H, I, g, seed):
    case = wl.MlpCase("t", M, H, I, g, seed, 0.005, 30.0)
    x = case.x()
    xb = wl.bf16_bits(x)
    Wg, Wu, Wd = case.W_gate().numpy(), case.W_up().numpy(), case.W_down().numpy()
    Wgu_q, sgu = oracle.quantize_weight(np.concatenate([Wg, Wu], 0), g)
    Wd_q, sd = oracle.quantize_weight(Wd, g)
    fused, _ = oracle.swiglu_mlp(xb, Wgu_q, sgu, None, Wd_q, sd, None, g)
    staged = oracle.staged_swiglu_mlp(xb, Wgu_q, sgu, None, Wd_q, sd, None, g)
    ref = oracle.reference_mlp_f64(oracle.bf16_bits_to_f32(xb), Wg, Wu, Wd)
    return (oracle.rel_l2(oracle.bf16_bits_to_f32(fused), ref),
            oracle.rel_l2(oracle.bf16_bits_to_f32(staged), ref))


def test_swiglu_mlp_error_levels_small():
    # at a small shape the fused/staged gap (~1e-4) is below sampling noise, so
    # only the INT8 noise level of both paths is pinned here
    e_fused, e_staged = _mlp_errors(128, 512, 256, 128, seed=21)
    assert 1e-3 < e_fused < 5e-2 and 1e-3 < e_staged < 5e-2
    assert abs(e_fused - e_staged) < 0.05 * e_staged


def test_fused_swiglu_error_no_worse_than_staged_mlp_2048_shape_rows():
    # the (2048, 3072 -> 1024) shape of the accuracy table, on 512 token rows
    # (rows are independent: per-token scales)
    e_fused, e_staged = _mlp_errors(512, 3072, 1024, 128, seed=4)
    assert e_fused <= e_staged


@pytest.mark.slow
def test_fused_swiglu_error_no_worse_than_staged_i12288_rows():
    # the (4096, 12288 -> 4096) entry of the accuracy table read literally
    # (hidden 4096, intermediate 12288), on 256 token rows
    e_fused, e_staged = _mlp_errors(256, 4096, 12288, 128, seed=3)
    assert e_fused <= e_staged


# --------------------------------------------------------------------------
# GEMV-resident layout (comfy-kitchen PR #248, Description)
# --------------------------------------------------------------------------

def _read_pack_fixture():
    out = {}
    for line in open(os.path.join(GOLDEN, "gemv_pack_fragment_positions.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        lane, *pairs = line.split()
        out[int(lane)] = [tuple(int(v) for v in p.split(",")) for p in pairs]
    return out


def test_gemv_pack_matches_hand_worked_fragment_positions():
    # a marker code at (row, col) must land at the fixture's byte of its lane
    fixture = _read_pack_fixture()
    sw = np.ones(16, np.float32)
    for lane, pos in fixture.items():
        for j, (r, c) in enumerate(pos):
            W = np.zeros((16, 32), np.int8)
            W[r, c] = 77
            packed = oracle.pack_gemv(W, sw)
            assert packed[16 * lane + j] == 77, (lane, j, r, c)
            assert np.count_nonzero(packed[:512]) == 1


def test_gemv_pack_is_a_bijection_per_block_and_interleaves_scales():
    N, K = 20, 64  # two 16-row tiles (second one padded), two 32-column blocks
    rng = np.random.default_rng(3)
    seen = {}
    sw = rng.random(N).astype(np.float32) + 0.5
    for r in range(16):
        for c in range(32):
            W = np.zeros((N, K), np.int8)
            W[r, 32 + c] = 1     # block 1 of tile 0
            W[16 + r % 4, c] = 2  # tile 1 (rows 16..19 exist)
            p = oracle.pack_gemv(W, sw)
            tile_bytes = 2 * 512 + 64
            hits = np.flatnonzero(p[:2 * 512] == 1)
            assert len(hits) == 1 and 512 <= hits[0] < 1024
            seen[(r, c)] = int(hits[0])
            assert np.count_nonzero(p[tile_bytes:tile_bytes + 1024] == 2) == 1
    assert sorted(seen.values()) == list(range(512, 1024))
    p = oracle.pack_gemv(np.zeros((N, K), np.int8), sw)
    tile_bytes = 2 * 512 + 64
    np.testing.assert_array_equal(p[1024:1088].view(np.float32), sw[:16])
    np.testing.assert_array_equal(p[tile_bytes + 1024:tile_bytes + 1088].view(np.float32)[:4],
                                  sw[16:])
    assert not p[tile_bytes + 1024 + 16:].any()  # padded rows: zero scales
    assert p.size == 2 * tile_bytes
