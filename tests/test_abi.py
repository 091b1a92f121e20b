"""The C ABI without a GPU: the library builds for sm_103a, loads, exports every
entry point include/ck.h declares, and rejects bad arguments with the right
status before touching the device.  No call here launches a kernel: each one
fails host-side validation first (fake pointers are never dereferenced)."""
import os
import re

import pytest
import torch

import swiglu_mlp_group_gb300 as ck

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ck.h")

# a fake, 16-byte aligned device address: validation rejects every call below
# before any pointer is used
P = 0x10000


@pytest.fixture(scope="module")
def L():
    ck.build()
    return ck.lib()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"CK_API\s+[^;(]*?\b(ck_\w+)\s*\(", text)


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 15
    for name in names:
        assert hasattr(L, name), name
    # and the binding exposes the same names
    for name in names:
        assert callable(getattr(ck, name)), name


def declared_parameter_counts():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"CK_API\s+[^;(]*?\b(ck_\w+)\s*\(([^)]*)\)", text):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else len(params.split(","))
    return out


def test_binding_argument_lists_match_the_header():
    # a positional mismatch would hand the library wrong pointers: every ctypes
    # signature of the binding must have the header's parameter count
    counts = declared_parameter_counts()
    assert len(counts) >= 15
    for name, (_, argtypes) in ck._SIGNATURES.items():
        assert name in counts, name
        assert len(argtypes) == counts[name], (name, len(argtypes), counts[name])
    assert set(counts) == set(ck._SIGNATURES)


def test_status_strings(L):
    for st in range(11):
        s = ck.status_string(st)
        assert s.startswith("CK_")
    assert ck.status_string(ck.CK_ERR_GROUP).startswith("CK_ERR_GROUP")
    assert L.ck_version() == 205


def test_workspace_and_prepared_sizes(L):
    M, K, N = 2048, 3072, 1024
    ws = ck.workspace_bytes(ck.CK_OP_INT8_LINEAR, M, K, N, ck.CK_WLAYOUT_GEMM_F16)
    assert ws >= M * K * 2 + M * 4
    ws_i8 = ck.workspace_bytes(ck.CK_OP_INT8_LINEAR, M, K, N, ck.CK_WLAYOUT_ROWMAJOR_I8)
    assert ws_i8 >= ws + N * K * 2
    assert L.ck_prepared_weight_bytes(ck.CK_WLAYOUT_GEMM_F16, N, K) == N * K * 2
    assert L.ck_prepared_weight_bytes(ck.CK_WLAYOUT_ROWMAJOR_I8, N, K) == N * K
    # GEMV layout: per 16-row tile, K/32 blocks of 512 bytes + 16 f32 scales
    assert L.ck_prepared_weight_bytes(ck.CK_WLAYOUT_GEMV_PACKED, 20, 64) == 2 * (2 * 512 + 64)
    assert L.ck_prepared_weight_bytes(ck.CK_WLAYOUT_GEMV_PACKED, 16, 48) == 0
    assert L.ck_prepared_weight_bytes(7, 16, 64) == 0
    # W6 / W4 GEMV layouts: blocks of 384 / 256 bytes, the same 64 scale bytes
    assert L.ck_prepared_weight_bytes(ck.CK_WLAYOUT_GEMV_PACKED_W6, 20, 64) == 2 * (2 * 384 + 64)
    assert L.ck_prepared_weight_bytes(ck.CK_WLAYOUT_GEMV_PACKED_W4, 20, 64) == 2 * (2 * 256 + 64)
    assert L.ck_prepared_weight_bytes(ck.CK_WLAYOUT_GEMV_PACKED_W4, 16, 48) == 0
    # interleaved gate|up: fp16 codes, an even number of rows
    assert L.ck_prepared_weight_bytes(ck.CK_WLAYOUT_GEMM_F16_GLU, 2 * 40, 64) == 80 * 64 * 2
    assert L.ck_prepared_weight_bytes(ck.CK_WLAYOUT_GEMM_F16_GLU, 41, 64) == 0
    assert (ck.workspace_bytes(ck.CK_OP_SWIGLU_MLP, 64, 256, 128, ck.CK_WLAYOUT_GEMM_F16_GLU)
            == ck.workspace_bytes(ck.CK_OP_SWIGLU_MLP, 64, 256, 128, ck.CK_WLAYOUT_GEMM_F16))
    assert ck.workspace_bytes(ck.CK_OP_INT8_LINEAR, 0, K, N) == 0


def lin(L, **kw):
    a = dict(x=P, M=64, K=256, ldx=256, act=0, W=P, wl=ck.CK_WLAYOUT_GEMM_F16, sw=P, N=128, g=64,
             bias=None, res=None, y=P, ws=P, ws_bytes=1 << 30, s=None)
    a.update(kw)
    return L.ck_int8_linear(a["x"], a["M"], a["K"], a["ldx"], a["act"], a["W"], a["wl"], a["sw"],
                            a["N"], a["g"], a["bias"], a["res"], a["y"], a["ws"], a["ws_bytes"],
                            a["s"])


def test_linear_validation_errors(L):
    assert lin(L, x=None) == ck.CK_ERR_NULL
    assert lin(L, W=None) == ck.CK_ERR_NULL
    assert lin(L, sw=None) == ck.CK_ERR_NULL
    assert lin(L, y=None) == ck.CK_ERR_NULL
    assert lin(L, act=5) == ck.CK_ERR_INVALID
    assert lin(L, wl=ck.CK_WLAYOUT_GEMV_PACKED) == ck.CK_ERR_INVALID
    assert lin(L, M=0) == ck.CK_ERR_SHAPE
    assert lin(L, K=0) == ck.CK_ERR_SHAPE
    assert lin(L, K=32768 + 256, ldx=32768 + 256) == ck.CK_ERR_SHAPE
    assert lin(L, ldx=128) == ck.CK_ERR_SHAPE              # ldx < K
    assert lin(L, ldx=260) == ck.CK_ERR_SHAPE              # ldx % 8
    assert lin(L, act=ck.CK_ACT_SWIGLU) == ck.CK_ERR_SHAPE  # swiglu needs ldx >= 2K
    assert lin(L, N=12) == ck.CK_ERR_SHAPE                 # N % 8
    assert lin(L, g=32) == ck.CK_ERR_GROUP
    assert lin(L, g=96) == ck.CK_ERR_GROUP
    assert lin(L, K=320, ldx=320, g=128) == ck.CK_ERR_GROUP  # K % g
    assert lin(L, x=P + 4) == ck.CK_ERR_ALIGN
    assert lin(L, y=P + 2) == ck.CK_ERR_ALIGN
    assert lin(L, bias=P + 8) == ck.CK_ERR_ALIGN
    assert lin(L, res=P + 8) == ck.CK_ERR_ALIGN
    assert lin(L, ws=None) == ck.CK_ERR_WORKSPACE
    assert lin(L, ws_bytes=100) == ck.CK_ERR_WORKSPACE


def test_other_entry_points_validate(L):
    assert L.ck_convrot_quantize_weight(None, 0, 8, 64, 64, P, P, None) == ck.CK_ERR_NULL
    assert L.ck_convrot_quantize_weight(P, 9, 8, 64, 64, P, P, None) == ck.CK_ERR_DTYPE
    assert L.ck_convrot_quantize_weight(P, 0, 8, 96, 64, P, P, None) == ck.CK_ERR_GROUP
    assert L.ck_convrot_quantize_weight(P, 0, 0, 64, 64, P, P, None) == ck.CK_ERR_SHAPE
    assert L.ck_rotate_quantize_act(P, 4, 256, 256, 3, 64, P, P, None) == ck.CK_ERR_INVALID
    assert L.ck_rotate_quantize_act(P, 4, 256, 256, 1, 64, P, P, None) == ck.CK_ERR_SHAPE
    assert L.ck_rotate_quantize_act(P, 4, 256, 256, 0, 512, P, P, None) == ck.CK_ERR_GROUP
    assert L.ck_prepare_weight(P, P, 16, 64, 9, P, 1 << 20, None) == ck.CK_ERR_INVALID
    assert L.ck_prepare_weight(P, P, 16, 48, 1, P, 1 << 20, None) == ck.CK_ERR_SHAPE
    assert L.ck_prepare_weight(P, P, 16, 64, 1, P, 10, None) == ck.CK_ERR_WORKSPACE
    assert L.ck_prepare_weight(P, None, 16, 64, 2, P, 1 << 20, None) == ck.CK_ERR_NULL
    assert (L.ck_int8_gemv_smallM(P, 9, 256, 256, 0, P, 128, 64, None, None, P, P, 1 << 20, None)
            == ck.CK_ERR_SHAPE)
    assert (L.ck_int8_gemv_smallM(P, 2, 256, 256, 0, P, 128, 64, None, P + 4, P, P, 1 << 20,
                                  None) == ck.CK_ERR_ALIGN)
    assert (L.ck_swiglu_mlp(P, 64, 256, 128, P, P, None, P, P, None, None, 1, 64, P, P, 10, None)
            == ck.CK_ERR_WORKSPACE)
    assert (L.ck_swiglu_mlp(P, 64, 256, 100, P, P, None, P, P, None, None, 1, 64, P, P, 1 << 30,
                            None) == ck.CK_ERR_GROUP)
    assert (L.ck_swiglu_mlp(P, 64, 256, 128, P, P, None, P, P, None, P + 2, 1, 64, P, P, 1 << 30,
                            None) == ck.CK_ERR_ALIGN)
    assert (L.ck_int8_gemm_dequant(P, P, 64, 256, P, P, 128, None, P + 8, P, None)
            == ck.CK_ERR_ALIGN)
    assert (L.ck_int8_gemv_dequant(P, P, 2, 256, P, 128, None, P + 8, P, None)
            == ck.CK_ERR_ALIGN)
    assert L.ck_debug_int8_gemm_s32(P, P, 8, 8, 96, P, P, 1 << 20, None) == ck.CK_ERR_SHAPE
    assert L.ck_prepare_weight(P, None, 41, 64, ck.CK_WLAYOUT_GEMM_F16_GLU, P, 1 << 20,
                               None) == ck.CK_ERR_SHAPE
    assert lin(L, wl=ck.CK_WLAYOUT_GEMM_F16_GLU) == ck.CK_ERR_INVALID  # MLP-only layout
    assert L.ck_debug_gemv_s32(P, 2, 256, P, ck.CK_WLAYOUT_GEMM_F16, 128, P, None) == ck.CK_ERR_INVALID
    assert L.ck_debug_gemv_s32(P, 9, 256, P, ck.CK_WLAYOUT_GEMV_PACKED, 128, P, None) == ck.CK_ERR_SHAPE
    assert L.ck_debug_gemv_s32(P, 2, 256, P, ck.CK_WLAYOUT_GEMV_PACKED, 12, P, None) == ck.CK_ERR_SHAPE
    assert L.ck_debug_gemv_s32(None, 2, 256, P, ck.CK_WLAYOUT_GEMV_PACKED, 128, P, None) == ck.CK_ERR_NULL
    # the W6A8 / W4A8 pieces
    for bits in (0, 5, 7, 9):
        assert L.ck_convrot_quantize_weight_bits(P, 0, 8, 64, 64, bits, P, P, None) == ck.CK_ERR_INVALID
    assert L.ck_convrot_quantize_weight_bits(None, 0, 8, 64, 64, 4, P, P, None) == ck.CK_ERR_NULL
    assert L.ck_convrot_quantize_weight_bits(P, 0, 8, 96, 64, 6, P, P, None) == ck.CK_ERR_GROUP
    assert L.ck_prepare_weight(P, None, 16, 64, ck.CK_WLAYOUT_GEMV_PACKED_W4, P, 1 << 20,
                               None) == ck.CK_ERR_NULL
    assert L.ck_prepare_weight(P, P, 16, 64, ck.CK_WLAYOUT_GEMV_PACKED_W6, P, 2 * 384 + 63,
                               None) == ck.CK_ERR_WORKSPACE
    for bad in (ck.CK_WLAYOUT_ROWMAJOR_I8, ck.CK_WLAYOUT_GEMM_F16, 5):
        assert (L.ck_packed_gemv_smallM(P, 2, 256, 256, 0, P, bad, 128, 64, None, None, P, P,
                                        1 << 20, None) == ck.CK_ERR_INVALID)
        assert (L.ck_packed_gemv_dequant(P, P, 2, 256, P, bad, 128, None, None, P, None)
                == ck.CK_ERR_INVALID)
    assert (L.ck_packed_gemv_smallM(P, 9, 256, 256, 0, P, ck.CK_WLAYOUT_GEMV_PACKED_W4, 128, 64,
                                    None, None, P, P, 1 << 20, None) == ck.CK_ERR_SHAPE)
    assert (L.ck_packed_gemv_dequant(P, P, 2, 256, P, ck.CK_WLAYOUT_GEMV_PACKED_W6, 128, None,
                                     P + 8, P, None) == ck.CK_ERR_ALIGN)


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_device_errors_without_a_gpu(L):
    assert L.ck_device_check() == ck.CK_ERR_UNSUPPORTED_DEVICE
    # fully valid arguments reach the device check, which fails: nothing launches
    assert lin(L) == ck.CK_ERR_UNSUPPORTED_DEVICE
    with pytest.raises(ck.CkError):
        ck._check(lin(L), "ck_int8_linear")


# The GEMM engine's variant choice (host logic): on the workloads' shapes it
# takes the variant measured fastest on a 152-SM GB300 (CUDA graphs, rotating
# inputs; times in microseconds, best first; 2048 x 1024 -> 3072 picks the
# 224-column pairs at 17.9 against one-SM 128 x 128 tiles at 18.6).
@pytest.mark.parametrize("M,N,K,code", [
    (4096, 4096, 4096, 448),     # 224-col pairs 73.7, 256-col pairs 81.5, one-SM 256 95.2
    (4096, 24576, 3072, 448),    # 306.2; 256-col pairs 316.0, one-SM 256 350.7
    (4096, 3072, 12288, 448),    # 154.7; 256-col pairs 171.1, one-SM 256 209.9
    (4096, 9216, 3072, 448),     # 119.0; 256-col pairs 121.5, one-SM 256 139.9
    (2048, 1024, 3072, 2128),    # 128-col pairs 16.3; one-SM 128 17.4, 224-col pairs 19.4
    (2048, 3072, 1024, 448),     # K = 1024: 224-col pairs 17.9, one-SM 128 18.6, 128-col pairs 18.7
    (2048, 2048, 3072, 512),     # 256-col pairs 22.8; one-SM 256 23.1, 128-col pairs 27.0
    (1024, 4096, 4096, 448),     # 24.6; 256-col pairs 27.1, one-SM 256 27.2
    (1024, 1024, 4096, 2128),    # 128-col pairs 18.1; one-SM 64 19.6, 224-col pairs 22.3
    (512, 3072, 3072, 2128),     # 15.6; 224-col pairs 18.7, 256-col pairs 21.3
    (256, 9216, 3072, 2128),     # 16.5; 224-col pairs 19.0, 256-col pairs 21.6
    (1024, 2048, 2048, 2128),    # 12.7; 224-col pairs 15.2, 256-col pairs 17.2
    (1, 128, 256, 128),
    (2048, 1024, 12288, 4512),   # K split between two pairs 37.0; 128-col pairs 44.7
    (512, 3072, 12288, 4512),    # 24 tiles of 256 x 256, K = 12288
    (2048, 2048, 12288, 512),    # 64 tiles of 256 x 256: their clusters do not all fit at once
])
def test_gemm_tile_choice_on_the_workload_shapes(L, M, N, K, code):
    assert ck.debug_gemm_tile_choice(M, N, K, 152) == code


def test_gemm_tile_choice_follows_the_forced_code_and_rejects_bad_sizes(L):
    ck.debug_force_gemm_tile(64)
    try:
        assert ck.debug_gemm_tile_choice(4096, 4096, 4096, 152) == 64
    finally:
        ck.debug_force_gemm_tile(0)
    assert ck.debug_gemm_tile_choice(4096, 4096, 4096, 152) == 448
    assert ck.debug_gemm_tile_choice(0, 4096, 4096, 152) == 0
    assert ck.debug_gemm_tile_choice(4096, 4096, 4096, 1) == 0
