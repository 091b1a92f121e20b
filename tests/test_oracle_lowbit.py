"""Pins for the oracle's W4A8 / W6A8 pieces (comfy-kitchen PR #248, "Performance
improvements for qwen 3.x (Part 2)", Commits and Description name 4- and 6-bit
weight decode; the formats are the reading stated in oracle/convrot_oracle.c):
the b-bit per-row quantizer against hand-worked rows, invariants, the textbook
g = 1 case and the INT8 quantizer at b = 8; the packed layouts against the
already pinned INT8 fragment layout, bit field by bit field, including the
claim that a code in the top bits of an INT8 lane is the INT8 value
code * 2^(8 - b); the low-bit linear against the closed-form error bound.
CPU only."""
import os

import numpy as np
import pytest

import oracle
from swiglu_mlp_group_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_fixture():
    cases, cur = [], {}
    for line in open(os.path.join(GOLDEN, "quantize_lowbit_rows.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        cur[key] = [float(v) for v in vals]
        if key == "codes":
            cases.append(cur)
            cur = {}
    return cases


def test_lowbit_quantizer_hand_worked_rows():
    cases = _read_fixture()
    assert len(cases) == 5
    for case in cases:
        bits = int(case["bits"][0])
        q, s = oracle.quantize_rows_bits(np.array([case["row"]], np.float32), bits)
        np.testing.assert_array_equal(q[0], np.array(case["codes"], np.int8))
        assert s[0] == np.float32(case["scale"][0])


@pytest.mark.parametrize("bits", [4, 6])
def test_lowbit_quantizer_invariants(bits):
    qmax = (1 << (bits - 1)) - 1
    v = wl.weight(120, 256, seed=40 + bits).numpy() * np.float32(3.0)
    v[5] = 0.0
    v[6] = -0.75
    q, s = oracle.quantize_rows_bits(v, bits)
    assert np.max(np.abs(q.astype(np.int32))) <= qmax
    for r in range(v.shape[0]):
        if r == 5:
            assert s[r] == 0.0 and not q[r].any()
            continue
        k = int(np.argmax(np.abs(v[r])))
        assert abs(int(q[r, k])) == qmax and np.sign(q[r, k]) == np.sign(v[r, k])
        assert s[r] == np.float32(np.max(np.abs(v[r]))) / np.float32(qmax)
    err = np.abs(v.astype(np.float64) - q.astype(np.float64) * s[:, None].astype(np.float64))
    assert np.all(err <= s[:, None].astype(np.float64) * (0.5 + 1e-5))
    assert np.all(q[6] == -qmax)


@pytest.mark.parametrize("bits", [4, 6])
def test_lowbit_group_one_is_textbook_rowwise_symmetric(bits):
    # g = 1: H is the identity; plain per-row absmax/qmax rounding written
    # independently with numpy (np.rint rounds half to even)
    qmax = (1 << (bits - 1)) - 1
    v = wl.weight(17, 64, seed=50 + bits).numpy() * np.float32(4.0)
    q, s = oracle.quantize_weight_bits(v, 1, bits)
    s_ref = (np.max(np.abs(v), axis=1) / np.float32(qmax)).astype(np.float32)
    q_ref = np.clip(np.rint(v / s_ref[:, None]), -qmax, qmax).astype(np.int8)
    np.testing.assert_array_equal(s, s_ref)
    np.testing.assert_array_equal(q, q_ref)


def test_lowbit_quantizer_at_8_bits_is_the_int8_quantizer():
    v = wl.weight(33, 128, seed=60).numpy() * np.float32(2.0)
    q8, s8 = oracle.quantize_rows(v)
    q, s = oracle.quantize_rows_bits(v, 8)
    np.testing.assert_array_equal(q, q8)
    np.testing.assert_array_equal(s, s8)


def _fragment_byte_of(r, c):
    """(lane, j) of code (r, c) of a 16 x 32 block in the pinned INT8 layout."""
    W = np.zeros((16, 32), np.int8)
    W[r, c] = 1
    hit = int(np.flatnonzero(oracle.pack_gemv(W, np.ones(16, np.float32))[:512])[0])
    return hit // 16, hit % 16


def _lane_byte_offsets(bits, lane):
    """Offsets in a block of the lane's bytes 0 .. 2 bits - 1: words 0 and 1
    at 8 lane, word 2 (6-bit) at 256 + 4 lane."""
    at = [8 * lane + p for p in range(8)]
    if bits == 6:
        at += [256 + 4 * lane + p for p in range(4)]
    return np.array(at)


def test_lowbit_lane_words_tile_the_block():
    """The lanes' words cover each block byte exactly once."""
    for bits in (4, 6):
        at = np.concatenate([_lane_byte_offsets(bits, l) for l in range(32)])
        assert sorted(at.tolist()) == list(range(64 * bits))


@pytest.mark.parametrize("bits", [4, 6])
def test_lowbit_pack_bit_fields_follow_the_int8_fragment_positions(bits):
    """Every code of a block, alone and negative, lands in exactly the bit
    field the stated layout gives for its INT8 fragment byte, and shifted into
    the top bits of a byte it reads back as code * 2^(8 - bits)."""
    code = -3 if bits == 4 else -21
    u = code & ((1 << bits) - 1)
    block_bytes = 64 * bits
    for r in range(16):
        for c in range(32):
            W = np.zeros((16, 32), np.int8)
            W[r, c] = code
            p = oracle.pack_gemv_lowbit(W, np.ones(16, np.float32), bits)
            blk = p[:block_bytes]
            lane, j = _fragment_byte_of(r, c)
            at = _lane_byte_offsets(bits, lane)
            lp = blk[at].astype(np.int64)
            others = np.delete(blk, at)
            assert not others.any(), (r, c)
            if bits == 4:
                byte = 4 * (j // 8) + j % 4
                shift = 4 * ((j // 4) % 2)
                assert (lp[byte] >> shift) & 0xF == u
                assert np.count_nonzero(lp) == 1
                as_int8 = np.int8(np.uint8((lp[byte] >> shift << 4) & 0xF0).view(np.int8))
            else:
                if j < 12:
                    byte = 4 * (j // 4) + j % 4
                    assert lp[byte] >> 2 == u and np.count_nonzero(lp) == 1
                    as_int8 = np.uint8(lp[byte] & 0xFC).view(np.int8)
                else:
                    i = j - 12
                    pieces = [lp[4 * w + i] & 3 for w in range(3)]
                    assert pieces[0] | pieces[1] << 2 | pieces[2] << 4 == u
                    assert np.count_nonzero(lp & 0xFC) == 0
                    as_int8 = np.uint8((pieces[0] | pieces[1] << 2 | pieces[2] << 4) << 2).view(np.int8)
            assert int(as_int8) == code * (1 << (8 - bits))


@pytest.mark.parametrize("bits", [4, 6])
def test_lowbit_pack_tiles_and_scales(bits):
    N, K = 20, 64
    rng = np.random.default_rng(bits)
    qmax = (1 << (bits - 1)) - 1
    W = rng.integers(-qmax, qmax + 1, size=(N, K)).astype(np.int8)
    sw = rng.random(N).astype(np.float32) + 0.5
    p = oracle.pack_gemv_lowbit(W, sw, bits)
    tile = 2 * 64 * bits + 64
    assert p.size == 2 * tile
    np.testing.assert_array_equal(p[2 * 64 * bits:tile].view(np.float32), sw[:16])
    np.testing.assert_array_equal(p[tile + 2 * 64 * bits:].view(np.float32)[:4], sw[16:])
    assert not p[tile + 2 * 64 * bits + 16:].any()
    # the padded rows 20..31 of tile 1 hold zero codes: re-packing with them
    # nonzero changes nothing in tile 0
    W2 = np.concatenate([W, np.ones((12, K), np.int8)], 0)
    p2 = oracle.pack_gemv_lowbit(W2, np.concatenate([sw, np.ones(12, np.float32)]), bits)
    np.testing.assert_array_equal(p2[:tile], p[:tile])


@pytest.mark.parametrize("bits", [4, 6])
def test_lowbit_linear_error_bound_closed_form(bits):
    """|y - y_ref| <= sum_k (|x_rot| sw/2 + |W_rot| sx/2 + 3 sx sw/4) + output
    rounding: the W8A8 bound with the b-bit step sw = absmax / qmax."""
    c = wl.LINEAR_TINY
    x, W, b = c.x(), c.W().numpy(), c.b()
    xb, bb = wl.bf16_bits(x), wl.bf16_bits(b)
    Wq, sw = oracle.quantize_weight_bits(W, c.g, bits)
    y = oracle.bf16_bits_to_f32(oracle.int8_linear(xb, Wq, sw, c.g, bb)).astype(np.float64)
    y_ref = oracle.reference_linear_f64(oracle.bf16_bits_to_f32(xb), W, oracle.bf16_bits_to_f32(bb))
    xq, sx = oracle.rotate_quantize_act(xb, c.g)
    xr = np.abs(oracle.rotate_rows(oracle.bf16_bits_to_f32(xb), c.g).astype(np.float64))
    wr = np.abs(oracle.rotate_rows(W, c.g).astype(np.float64))
    sx64, sw64 = sx.astype(np.float64)[:, None], sw.astype(np.float64)[None, :]
    bound = (xr.sum(1)[:, None] * sw64 / 2 + wr.sum(1)[None, :] * sx64 / 2 + 0.75 * c.K * sx64 * sw64)
    bound += 1e-5 * (xr @ wr.T) + np.abs(y_ref) * 2.0 ** -8 + 1e-30
    assert np.all(np.abs(y - y_ref) <= bound)
    # coarser grids, larger error: 4-bit above 6-bit above 8-bit
    e = oracle.rel_l2(y, y_ref)
    Wq8, sw8 = oracle.quantize_weight(W, c.g)
    e8 = oracle.rel_l2(oracle.bf16_bits_to_f32(oracle.int8_linear(xb, Wq8, sw8, c.g, bb)), y_ref)
    assert e > e8
