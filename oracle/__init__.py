"""CPU oracle for the ConvRot INT8 W8A8 linear and the fused SwiGLU MLP.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers.  The product library
(``swiglu_mlp_group_gb300``) never imports this package, and this package
never imports the product library: the two share no code.

The arithmetic lives in ``convrot_oracle.c`` (plain C, float64 / int64).  This
module builds it with gcc on first use, loads it with ctypes, and composes the
steps into the method's calls.  bf16 values cross this interface as their raw
16-bit patterns in ``numpy.uint16`` arrays.

Sources (web pages; cited by title and section):
  [P1] sglang PR #44196, "comfy_kitchen SwiGLU MLP for Qwen-Image 2.1"
  [P3] sglang PR #35994 report, "Load serialized Comfy ConvRot INT8 DiTs"
  [P4] comfy-kitchen PR #277, "FP16 tensor-core fallback for int8_linear"

Parity status: every function here is pinned by ``tests/test_oracle.py``
against closed forms, textbook special cases, brute force or invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "convrot_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

_c_i64 = ctypes.c_int64
_ptr = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the C oracle into oracle/_build/liboracle.so (gcc, OpenMP).

    ``-ffp-contract=off`` keeps gcc from fusing multiply-adds (it would on
    aarch64 by default), so the float64 arithmetic is the same on every host.
    """
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-shared",
           "-fPIC", "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oracle_sylvester_hadamard.argtypes = [ctypes.c_int, _ptr]
        lib.oracle_sylvester_hadamard.restype = ctypes.c_int
        lib.oracle_rotate_rows_f64.argtypes = [_ptr, _c_i64, _c_i64, _c_i64, ctypes.c_int, _ptr]
        lib.oracle_rotate_rows_f64.restype = ctypes.c_int
        lib.oracle_rotate_rows.argtypes = [_ptr, _c_i64, _c_i64, _c_i64, ctypes.c_int, _ptr]
        lib.oracle_rotate_rows.restype = ctypes.c_int
        lib.oracle_quantize_rows.argtypes = [_ptr, _c_i64, _c_i64, _ptr, _ptr]
        lib.oracle_quantize_rows.restype = None
        lib.oracle_swiglu.argtypes = [_ptr, _c_i64, _c_i64, _c_i64, _ptr]
        lib.oracle_swiglu.restype = None
        lib.oracle_int8_gemm.argtypes = [_ptr, _ptr, _c_i64, _c_i64, _c_i64, _ptr]
        lib.oracle_int8_gemm.restype = None
        lib.oracle_f32_to_bf16_bits.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_bf16_bits.restype = ctypes.c_uint16
        lib.oracle_bf16_bits_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_bits_to_f32.restype = ctypes.c_float
        lib.oracle_dequant.argtypes = [_ptr, _ptr, _ptr, _ptr, _ptr, _c_i64, _c_i64, _ptr]
        lib.oracle_dequant.restype = None
        lib.oracle_round_to_bf16.argtypes = [_ptr, _c_i64, _ptr]
        lib.oracle_round_to_bf16.restype = None
        lib.oracle_pack_gemv.argtypes = [_ptr, _ptr, _c_i64, _c_i64, _ptr]
        lib.oracle_pack_gemv.restype = None
        lib.oracle_quantize_rows_bits.argtypes = [_ptr, _c_i64, _c_i64, ctypes.c_int, _ptr, _ptr]
        lib.oracle_quantize_rows_bits.restype = None
        lib.oracle_pack_gemv_lowbit.argtypes = [_ptr, _ptr, _c_i64, _c_i64, ctypes.c_int, _ptr]
        lib.oracle_pack_gemv_lowbit.restype = ctypes.c_int
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        lib.oracle_set_num_threads.restype = None
        _lib = lib
        return lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=dtype))


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


# --------------------------------------------------------------------------
# Elementary steps (each a thin call into the C oracle)
# --------------------------------------------------------------------------

def hadamard(g: int) -> np.ndarray:
    """Normalised Sylvester Hadamard H_g (float64, g x g).  [P4] The key observation."""
    H = np.empty((g, g), dtype=np.float64)
    if _load().oracle_sylvester_hadamard(int(g), _p(H)) != 0:
        raise ValueError(f"group size {g} is not a power of two")
    return H


def rotate_rows_f64(v: np.ndarray, g: int) -> np.ndarray:
    """Block-diagonal group rotation in float64, no rounding.  [P4] x_rot = x @ H."""
    v = _c(v, np.float64)
    rows, K = v.shape
    out = np.empty_like(v)
    rc = _load().oracle_rotate_rows_f64(_p(v), rows, K, K, int(g), _p(out))
    if rc != 0:
        raise ValueError(f"rotate: bad group size {g} for K={K} (rc={rc})")
    return out


def rotate_rows(v: np.ndarray, g: int) -> np.ndarray:
    """Group rotation of f32 rows: float64 product, result rounded once to f32."""
    v = _c(v, np.float32)
    rows, K = v.shape
    out = np.empty_like(v)
    rc = _load().oracle_rotate_rows(_p(v), rows, K, K, int(g), _p(out))
    if rc != 0:
        raise ValueError(f"rotate: bad group size {g} for K={K} (rc={rc})")
    return out


def quantize_rows(v: np.ndarray):
    """Per-row absmax/127 INT8 codes (round half to even, clamp +-127) + f32 scales.

    [P3] kitchen_int8.py process_weights_after_loading (per_channel=True,
    stochastic_rounding=0); [P4] Notes for the reviewer (same grid for the
    activation).  Returns (codes int8 [rows, K], scale f32 [rows]).
    """
    v = _c(v, np.float32)
    rows, K = v.shape
    q = np.empty((rows, K), dtype=np.int8)
    s = np.empty((rows,), dtype=np.float32)
    _load().oracle_quantize_rows(_p(v), rows, K, _p(q), _p(s))
    return q, s


def swiglu(h: np.ndarray) -> np.ndarray:
    """a = f32(silu(gate) * up) from packed rows [gate | up] (f32).  [P1] Motivation."""
    h = _c(h, np.float32)
    rows, two_i = h.shape
    if two_i % 2:
        raise ValueError("swiglu input needs an even number of columns")
    I = two_i // 2
    a = np.empty((rows, I), dtype=np.float32)
    _load().oracle_swiglu(_p(h), rows, I, two_i, _p(a))
    return a


def int8_gemm(xq: np.ndarray, wq: np.ndarray) -> np.ndarray:
    """acc[m, n] = sum_k xq[m, k] * wq[n, k] in int64.  [P4] Summary."""
    xq = _c(xq, np.int8)
    wq = _c(wq, np.int8)
    M, K = xq.shape
    N, K2 = wq.shape
    if K != K2:
        raise ValueError("K mismatch")
    acc = np.empty((M, N), dtype=np.int64)
    _load().oracle_int8_gemm(_p(xq), _p(wq), M, N, K, _p(acc))
    return acc


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round f32 to bf16 (nearest, ties to even), returning the raw bits."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_round_to_bf16(_p(x), x.size, _p(out))
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to f32."""
    b = _c(b, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def dequant(acc: np.ndarray, sx: np.ndarray, sw: np.ndarray, bias_bits=None,
            residual_bits=None) -> np.ndarray:
    """y = bf16(f32(acc * sx[m] * sw[n] + bias[n] + residual[m, n])) with float64
    inside.  [P4] Summary; [P2] Commits (residual fused into the epilogue)."""
    acc = _c(acc, np.int64)
    sx = _c(sx, np.float32)
    sw = _c(sw, np.float32)
    M, N = acc.shape
    y = np.empty((M, N), dtype=np.uint16)
    b = None if bias_bits is None else _c(bias_bits, np.uint16)
    r = None if residual_bits is None else _c(residual_bits, np.uint16)
    if r is not None and r.shape != (M, N):
        raise ValueError("residual must be bf16 bits of shape [M, N]")
    _load().oracle_dequant(_p(acc), _p(sx), _p(sw), None if b is None else _p(b),
                           None if r is None else _p(r), M, N, _p(y))
    return y


def pack_gemv(Wq: np.ndarray, sw: np.ndarray) -> np.ndarray:
    """GEMV-resident layout of int8 codes [N, K] + f32 scales [N] (uint8 bytes).

    comfy-kitchen PR #248, Description (weights and scales interleaved); the
    page does not fix the tiling: the one used is stated in convrot_oracle.c.
    """
    Wq = _c(Wq, np.int8)
    sw = _c(sw, np.float32)
    N, K = Wq.shape
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    out = np.empty(((N + 15) // 16) * (K * 16 + 64), dtype=np.uint8)
    _load().oracle_pack_gemv(_p(Wq), _p(sw), N, K, _p(out))
    return out


def qmax_of_bits(bits: int) -> int:
    """Largest code magnitude of signed symmetric b-bit codes: 2^(b-1) - 1."""
    if bits not in (4, 6, 8):
        raise ValueError("weight codes of 4, 6 or 8 bits")
    return (1 << (bits - 1)) - 1


def quantize_rows_bits(v: np.ndarray, bits: int):
    """Per-row absmax/qmax codes of `bits` bits (qmax = 2^(bits-1) - 1), ties to
    even, clamp to [-qmax, qmax] -> (q int8 [rows, K], scale f32 [rows]).
    comfy-kitchen PR #248, Commits and Description (W4A8 / W6A8 weights; the
    format is this package's reading, stated in convrot_oracle.c)."""
    v = _c(v, np.float32)
    rows, K = v.shape
    q = np.empty((rows, K), dtype=np.int8)
    s = np.empty((rows,), dtype=np.float32)
    _load().oracle_quantize_rows_bits(_p(v), rows, K, qmax_of_bits(bits), _p(q), _p(s))
    return q, s


def pack_gemv_lowbit(Wq: np.ndarray, sw: np.ndarray, bits: int) -> np.ndarray:
    """GEMV-resident layout of 4- or 6-bit codes [N, K] + f32 scales [N] (uint8
    bytes; the bit positions are stated in convrot_oracle.c)."""
    Wq = _c(Wq, np.int8)
    sw = _c(sw, np.float32)
    N, K = Wq.shape
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    out = np.empty(((N + 15) // 16) * (K // 32 * 64 * bits + 64), dtype=np.uint8)
    if _load().oracle_pack_gemv_lowbit(_p(Wq), _p(sw), N, K, int(bits), _p(out)) != 0:
        raise ValueError("bits must be 4 or 6")
    return out


# --------------------------------------------------------------------------
# The method's calls, composed from the steps above
# --------------------------------------------------------------------------

def quantize_weight(W: np.ndarray, g: int):
    """Offline ConvRot weight quantization: W_rot = W @ H (per group), then per
    output row absmax/127 codes.  Returns (Wq int8 [N, K], sw f32 [N]).

    [P3] kitchen_int8.py process_weights_after_loading (TensorWiseINT8Layout
    .quantize with per_channel=True, convrot=True, convrot_groupsize=g,
    stochastic_rounding=0; F32 scale of shape [out_features, 1]).
    """
    return quantize_rows(rotate_rows(_c(W, np.float32), g))


def quantize_weight_bits(W: np.ndarray, g: int, bits: int):
    """Offline ConvRot weight quantization to b-bit codes (W4A8 / W6A8; bits = 8
    is quantize_weight): W_rot = W @ H per group, per-row absmax/qmax codes.
    Returns (Wq int8 [N, K] in [-qmax, qmax], sw f32 [N])."""
    return quantize_rows_bits(rotate_rows(_c(W, np.float32), g), bits)


def act_input_f32(x_bits: np.ndarray, act: str) -> np.ndarray:
    """The f32 row the activation quantizer rotates: the widened bf16 input
    (act='none') or f32(silu(gate) * up) of the packed [gate | up] input
    (act='swiglu', [P1] Motivation)."""
    x = bf16_bits_to_f32(x_bits)
    if act == "none":
        return x
    if act == "swiglu":
        return swiglu(x)
    raise ValueError(f"unknown input activation {act!r}")


def rotate_quantize_act(x_bits: np.ndarray, g: int, act: str = "none"):
    """Online per-token activation quantization: [swiglu ->] rotate -> absmax/127
    codes.  Returns (xq int8 [M, K], sx f32 [M]).  [P4] The key observation and
    Notes for the reviewer; [P1] Motivation for act='swiglu'."""
    return quantize_rows(rotate_rows(act_input_f32(x_bits, act), g))


def int8_linear(x_bits, Wq, sw, g: int, bias_bits=None, act: str = "none",
                residual_bits=None):
    """y = dequant(int8_gemm(quant(rot(x)), Wq)) (+ residual) as bf16 bits [M, N].

    [P4] The key observation: y = x @ W^T = x_rot @ W_rot^T, with the inverse
    rotation never applied.
    """
    xq, sx = rotate_quantize_act(x_bits, g, act)
    return dequant(int8_gemm(xq, Wq), sx, sw, bias_bits, residual_bits)


def swiglu_mlp(x_bits, Wgu_q, sgu, bgu_bits, Wd_q, sd, bd_bits, g: int, residual_bits=None):
    """Fused SwiGLU MLP: one packed [gate | up] linear, then the down linear whose
    quantizer applies silu(gate) * up in f32 (its epilogue adds the residual, if
    any).  [P1] Motivation / Modifications."""
    h_bits = int8_linear(x_bits, Wgu_q, sgu, g, bgu_bits, "none")
    return int8_linear(h_bits, Wd_q, sd, g, bd_bits, "swiglu", residual_bits), h_bits


def staged_swiglu_mlp(x_bits, Wgu_q, sgu, bgu_bits, Wd_q, sd, bd_bits, g: int):
    """The older eager path, for comparison only: silu(gate) and the product are
    each rounded to bf16 and written out before the down linear.  [P1]
    Motivation (silu(gate) * up written to HBM in BF16)."""
    h_bits = int8_linear(x_bits, Wgu_q, sgu, g, bgu_bits, "none")
    h = bf16_bits_to_f32(h_bits)
    I = h.shape[1] // 2
    gate = h[:, :I].astype(np.float64)
    up = h[:, I:]
    silu_bits = f32_to_bf16_bits((gate / (1.0 + np.exp(-gate))).astype(np.float32))
    a_bits = f32_to_bf16_bits(bf16_bits_to_f32(silu_bits) * up)
    return int8_linear(a_bits, Wd_q, sd, g, bd_bits, "none")


def reference_linear_f64(x: np.ndarray, W: np.ndarray, bias=None) -> np.ndarray:
    """Unquantized float64 reference y = x @ W^T (+ b), for error metrics."""
    y = np.asarray(x, np.float64) @ np.asarray(W, np.float64).T
    if bias is not None:
        y = y + np.asarray(bias, np.float64)[None, :]
    return y


def reference_mlp_f64(x, Wg, Wu, Wd, bg=None, bu=None, bd=None) -> np.ndarray:
    """Unquantized float64 SwiGLU MLP down(silu(x Wg^T) * (x Wu^T))."""
    gt = reference_linear_f64(x, Wg, bg)
    up = reference_linear_f64(x, Wu, bu)
    a = gt / (1.0 + np.exp(-gt)) * up
    return reference_linear_f64(a, Wd, bd)


def rel_l2(y, y_ref) -> float:
    """||y - y_ref||_2 / ||y_ref||_2 in float64."""
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    den = float(np.linalg.norm(y_ref))
    return float(np.linalg.norm(y - y_ref)) / (den if den > 0 else 1.0)
