"""GB300 (sm_103a) ConvRot INT8 W8A8 linear, fused SwiGLU MLP and small-M GEMV.

Python binding of the C ABI in ``include/ck.h`` (library ``libck_gb300.so``).
The ``ck_*`` functions below are the C entry points themselves (ctypes); the
lower-case helpers only marshal torch tensors (device memory, streams) into
those calls -- every step of the computation runs in the library's CUDA
kernels.  There is no CPU or PyTorch fallback: if the library is missing or the
device is not a GB300, the calls raise.

The method (web pages, cited by title and section): comfy-kitchen PR #277
"FP16 tensor-core fallback for int8_linear" (The key observation), sglang PR
#44196 "comfy_kitchen SwiGLU MLP for Qwen-Image 2.1" (Motivation), sglang PR
#35994 report "Load serialized Comfy ConvRot INT8 DiTs" (kitchen_int8.py
excerpt), comfy-kitchen PR #248 "Performance improvements for qwen 3.x
(Part 2)" (Description).
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "CkError", "lib", "library_path", "build",
    "CK_OK", "CK_ERR_NULL", "CK_ERR_SHAPE", "CK_ERR_DTYPE", "CK_ERR_GROUP", "CK_ERR_ALIGN",
    "CK_ERR_WORKSPACE", "CK_ERR_UNSUPPORTED_DEVICE", "CK_ERR_CUDA", "CK_ERR_TIMEOUT",
    "CK_ERR_INVALID", "CK_F32", "CK_BF16", "CK_ACT_NONE", "CK_ACT_SWIGLU",
    "CK_WLAYOUT_ROWMAJOR_I8", "CK_WLAYOUT_GEMM_F16", "CK_WLAYOUT_GEMV_PACKED",
    "CK_WLAYOUT_GEMV_PACKED_W6", "CK_WLAYOUT_GEMV_PACKED_W4", "CK_WLAYOUT_GEMM_F16_GLU",
    "GEMV_LAYOUT_OF_BITS",
    "CK_OP_INT8_LINEAR", "CK_OP_SWIGLU_MLP", "CK_OP_GEMV_SMALLM", "CK_OP_DEBUG_GEMM_S32",
    "quantize_weight", "rotate_quantize_act", "prepare_weight", "int8_linear", "swiglu_mlp",
    "gemv_smallM", "quantize_weight_bits", "packed_gemv_dequant", "debug_int8_gemm_s32", "poll_device_status", "set_wait_timeout_ns",
    "set_launch_overlap", "debug_stalled_wait", "workspace_bytes",
]

# ck_status
CK_OK, CK_ERR_NULL, CK_ERR_SHAPE, CK_ERR_DTYPE, CK_ERR_GROUP, CK_ERR_ALIGN = 0, 1, 2, 3, 4, 5
CK_ERR_WORKSPACE, CK_ERR_UNSUPPORTED_DEVICE, CK_ERR_CUDA, CK_ERR_TIMEOUT, CK_ERR_INVALID = (
    6, 7, 8, 9, 10)
# ck_dtype, ck_input_act, ck_wlayout, ck_op
CK_F32, CK_BF16 = 0, 1
CK_ACT_NONE, CK_ACT_SWIGLU = 0, 1
CK_WLAYOUT_ROWMAJOR_I8, CK_WLAYOUT_GEMM_F16, CK_WLAYOUT_GEMV_PACKED = 0, 1, 2
CK_WLAYOUT_GEMV_PACKED_W6, CK_WLAYOUT_GEMV_PACKED_W4, CK_WLAYOUT_GEMM_F16_GLU = 3, 4, 5
# the GEMV-resident layout of each weight code width
GEMV_LAYOUT_OF_BITS = {8: CK_WLAYOUT_GEMV_PACKED, 6: CK_WLAYOUT_GEMV_PACKED_W6,
                       4: CK_WLAYOUT_GEMV_PACKED_W4}
CK_OP_INT8_LINEAR, CK_OP_SWIGLU_MLP, CK_OP_GEMV_SMALLM, CK_OP_DEBUG_GEMM_S32 = 0, 1, 2, 3

_ACTS = {"none": CK_ACT_NONE, "swiglu": CK_ACT_SWIGLU}

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None

_i64, _vp, _sz, _int = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
# name -> (restype, argtypes), in the order of include/ck.h
_SIGNATURES = {
    "ck_status_string": (ctypes.c_char_p, [_int]),
    "ck_version": (_int, []),
    "ck_device_check": (_int, []),
    "ck_convrot_quantize_weight": (_int, [_vp, _int, _i64, _i64, _int, _vp, _vp, _vp]),
    "ck_convrot_quantize_weight_bits": (_int, [_vp, _int, _i64, _i64, _int, _int, _vp, _vp, _vp]),
    "ck_rotate_quantize_act": (_int, [_vp, _i64, _i64, _i64, _int, _int, _vp, _vp, _vp]),
    "ck_rotate_quantize_act_f16": (_int, [_vp, _i64, _i64, _i64, _int, _int, _vp, _vp, _vp]),
    "ck_int8_gemm_dequant": (_int, [_vp, _vp, _i64, _i64, _vp, _vp, _i64, _vp, _vp, _vp, _vp]),
    "ck_prepared_weight_bytes": (_sz, [_int, _i64, _i64]),
    "ck_prepare_weight": (_int, [_vp, _vp, _i64, _i64, _int, _vp, _sz, _vp]),
    "ck_workspace_bytes": (_sz, [_int, _i64, _i64, _i64, _int]),
    "ck_int8_linear": (_int, [_vp, _i64, _i64, _i64, _int, _vp, _int, _vp, _i64, _int, _vp, _vp,
                              _vp, _vp, _sz, _vp]),
    "ck_int8_linear_noalloc": (_int, [_vp, _i64, _i64, _i64, _int, _vp, _vp, _i64, _int, _vp, _vp,
                                      _vp, _vp]),
    "ck_swiglu_mlp": (_int, [_vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _int, _int,
                             _vp, _vp, _sz, _vp]),
    "ck_int8_gemv_smallM": (_int, [_vp, _i64, _i64, _i64, _int, _vp, _i64, _int, _vp, _vp, _vp,
                                   _vp, _sz, _vp]),
    "ck_int8_gemv_dequant": (_int, [_vp, _vp, _i64, _i64, _vp, _i64, _vp, _vp, _vp, _vp]),
    "ck_packed_gemv_smallM": (_int, [_vp, _i64, _i64, _i64, _int, _vp, _int, _i64, _int, _vp, _vp,
                                     _vp, _vp, _sz, _vp]),
    "ck_packed_gemv_dequant": (_int, [_vp, _vp, _i64, _i64, _vp, _int, _i64, _vp, _vp, _vp, _vp]),
    "ck_poll_device_status": (_int, [_vp]),
    "ck_set_wait_timeout_ns": (None, [ctypes.c_uint64]),
    "ck_set_launch_overlap": (None, [_int]),
    "ck_debug_int8_gemm_s32": (_int, [_vp, _vp, _i64, _i64, _i64, _vp, _vp, _sz, _vp]),
    "ck_measure_int8_mma_tops": (_int, [ctypes.POINTER(ctypes.c_double), _vp, _vp]),
    "ck_measure_tcgen05_f16_tflops": (_int, [ctypes.POINTER(ctypes.c_double), _vp]),
    "ck_debug_gemv_s32": (_int, [_vp, _i64, _i64, _vp, _int, _i64, _vp, _vp]),
    "ck_debug_force_gemm_tile": (None, [_int]),
    "ck_debug_gemm_tile_choice": (_int, [_i64, _i64, _i64, _int]),
    "ck_debug_force_gemv_quantizer": (None, [_int]),
    "ck_debug_stalled_wait": (_int, [_vp]),
}


class CkError(RuntimeError):
    """A ck_* call returned a status other than CK_OK."""

    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {status_string(status)}")


def library_path() -> str:
    from . import _build
    return _build.LIB_PATH


def build(force: bool = False) -> str:
    """Compile libck_gb300.so for sm_103a (nvcc); returns its path."""
    from . import _build
    return _build.build(force=force)


def lib():
    """The loaded library.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
        return _lib


def _make_entry(name):
    def entry(*args):
        return getattr(lib(), name)(*args)
    entry.__name__ = name
    entry.__doc__ = f"The C entry point {name} of include/ck.h (ctypes)."
    return entry


for _name in _SIGNATURES:
    globals()[_name] = _make_entry(_name)
    __all__.append(_name)


def status_string(st: int) -> str:
    return lib().ck_status_string(int(st)).decode()


def _check(st: int, where: str) -> None:
    if st != CK_OK:
        raise CkError(st, where)


# ---------------------------------------------------------------------------
# torch marshalling
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _stream(stream=None) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _check_residual(residual, M: int, N: int) -> None:
    """A residual must be a contiguous bf16 [M, N] tensor (the library reads rows of N)."""
    if residual is None:
        return
    torch = _torch()
    if residual.dtype != torch.bfloat16 or tuple(residual.shape) != (M, N) or \
            not residual.is_contiguous():
        raise ValueError(f"residual must be a contiguous bf16 tensor of shape ({M}, {N})")


def _require_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("expected contiguous CUDA tensors")


def workspace_bytes(op: int, M: int, K: int, N: int, wlayout: int = CK_WLAYOUT_GEMM_F16) -> int:
    return int(lib().ck_workspace_bytes(op, M, K, N, wlayout))


def _workspace(nbytes: int, device):
    torch = _torch()
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def quantize_weight(W, g: int, stream=None):
    """Offline ConvRot weight quantization -> (Wq int8 [N, K], sw f32 [N])."""
    torch = _torch()
    _require_cuda(W)
    N, K = W.shape
    wdt = {torch.float32: CK_F32, torch.bfloat16: CK_BF16}[W.dtype]
    Wq = torch.empty((N, K), dtype=torch.int8, device=W.device)
    sw = torch.empty((N,), dtype=torch.float32, device=W.device)
    _check(lib().ck_convrot_quantize_weight(W.data_ptr(), wdt, N, K, g, Wq.data_ptr(),
                                            sw.data_ptr(), _stream(stream)),
           "ck_convrot_quantize_weight")
    return Wq, sw


def quantize_weight_bits(W, g: int, bits: int, stream=None):
    """ConvRot weight quantization to b-bit codes (bits 8, 6 or 4: W8A8 / W6A8 /
    W4A8) -> (Wq int8 [N, K] within +-(2^(bits-1) - 1), sw f32 [N])."""
    torch = _torch()
    _require_cuda(W)
    N, K = W.shape
    wdt = {torch.float32: CK_F32, torch.bfloat16: CK_BF16}[W.dtype]
    Wq = torch.empty((N, K), dtype=torch.int8, device=W.device)
    sw = torch.empty((N,), dtype=torch.float32, device=W.device)
    _check(lib().ck_convrot_quantize_weight_bits(W.data_ptr(), wdt, N, K, g, int(bits), Wq.data_ptr(),
                                                 sw.data_ptr(), _stream(stream)),
           "ck_convrot_quantize_weight_bits")
    return Wq, sw


def rotate_quantize_act(x, g: int, act: str = "none", K: int | None = None, stream=None):
    """Online activation rotation + per-token quantization -> (xq int8 [M, K], sx f32 [M])."""
    torch = _torch()
    _require_cuda(x)
    M, ldx = x.shape
    if K is None:
        K = ldx // 2 if act == "swiglu" else ldx
    xq = torch.empty((M, K), dtype=torch.int8, device=x.device)
    sx = torch.empty((M,), dtype=torch.float32, device=x.device)
    _check(lib().ck_rotate_quantize_act(x.data_ptr(), M, K, ldx, _ACTS[act], g, xq.data_ptr(),
                                        sx.data_ptr(), _stream(stream)), "ck_rotate_quantize_act")
    return xq, sx


def rotate_quantize_act_f16(x, g: int, act: str = "none", K: int | None = None, stream=None):
    """Activation quantization with fp16-held codes -> (xq16 fp16 [M, K], sx f32 [M])."""
    torch = _torch()
    _require_cuda(x)
    M, ldx = x.shape
    if K is None:
        K = ldx // 2 if act == "swiglu" else ldx
    xq = torch.empty((M, K), dtype=torch.float16, device=x.device)
    sx = torch.empty((M,), dtype=torch.float32, device=x.device)
    _check(lib().ck_rotate_quantize_act_f16(x.data_ptr(), M, K, ldx, _ACTS[act], g, xq.data_ptr(),
                                            sx.data_ptr(), _stream(stream)),
           "ck_rotate_quantize_act_f16")
    return xq, sx


def int8_gemm_dequant(xq16, sx, W16, sw, bias=None, out=None, stream=None, residual=None):
    """GEMM + dequant on fp16-held codes and a CK_WLAYOUT_GEMM_F16 weight -> y bf16 [M, N]
    (+ residual bf16 [M, N], which may be `out` itself)."""
    torch = _torch()
    _require_cuda(xq16, sx, W16, sw, bias, residual)
    M, K = xq16.shape
    N = sw.shape[0]
    _check_residual(residual, M, N)
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=xq16.device)
    _check(lib().ck_int8_gemm_dequant(xq16.data_ptr(), sx.data_ptr(), M, K, W16.data_ptr(),
                                      sw.data_ptr(), N, _ptr(bias), _ptr(residual), y.data_ptr(),
                                      _stream(stream)),
           "ck_int8_gemm_dequant")
    return y


def measure_int8_mma_tops(stream=None) -> float:
    """Dense mma.sync s8 throughput of the current device (TOPS)."""
    torch = _torch()
    v = ctypes.c_double(0.0)
    sink = torch.zeros(4, dtype=torch.int32, device="cuda")
    _check(lib().ck_measure_int8_mma_tops(ctypes.byref(v), sink.data_ptr(), _stream(stream)),
           "ck_measure_int8_mma_tops")
    return v.value


def measure_tcgen05_f16_tflops(stream=None) -> float:
    """Issue rate of tcgen05.mma kind::f16 128x256x16 on the whole device (TFLOP/s)."""
    v = ctypes.c_double(0.0)
    _check(lib().ck_measure_tcgen05_f16_tflops(ctypes.byref(v), _stream(stream)),
           "ck_measure_tcgen05_f16_tflops")
    return v.value


def prepare_weight(Wq, sw, layout: int, stream=None):
    """Re-lay a quantized weight into a resident layout (a flat uint8 device tensor)."""
    torch = _torch()
    _require_cuda(Wq, sw)
    N, K = Wq.shape
    nbytes = int(lib().ck_prepared_weight_bytes(layout, N, K))
    if nbytes == 0:
        raise CkError(CK_ERR_SHAPE, "ck_prepared_weight_bytes")
    out = torch.empty((nbytes,), dtype=torch.uint8, device=Wq.device)
    _check(lib().ck_prepare_weight(Wq.data_ptr(), _ptr(sw), N, K, layout, out.data_ptr(), nbytes,
                                   _stream(stream)), "ck_prepare_weight")
    return out


def int8_linear(x, W, sw, g: int, bias=None, act: str = "none", N: int | None = None,
                wlayout: int = CK_WLAYOUT_ROWMAJOR_I8, out=None, workspace=None, stream=None,
                residual=None):
    """ConvRot W8A8 linear y = bf16(acc * sx * sw + bias + residual) -> y bf16 [M, N]."""
    torch = _torch()
    _require_cuda(x, W, sw, bias, residual)
    M, ldx = x.shape
    K = ldx // 2 if act == "swiglu" else ldx
    if N is None:
        N = sw.shape[0]
    _check_residual(residual, M, N)
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    need = workspace_bytes(CK_OP_INT8_LINEAR, M, K, N, wlayout)
    ws = workspace if workspace is not None else _workspace(need, x.device)
    _check(lib().ck_int8_linear(x.data_ptr(), M, K, ldx, _ACTS[act], W.data_ptr(), wlayout,
                                sw.data_ptr(), N, g, _ptr(bias), _ptr(residual), y.data_ptr(),
                                ws.data_ptr(), ws.numel(), _stream(stream)), "ck_int8_linear")
    return y


def swiglu_mlp(x, Wgu, sgu, Wd, sd, g: int, bgu=None, bd=None,
               wlayout: int = CK_WLAYOUT_ROWMAJOR_I8, out=None, workspace=None, stream=None,
               residual=None):
    """Fused SwiGLU MLP: packed [gate | up] linear, then the swiglu-quantized down linear
    (whose epilogue adds `residual`, bf16 [M, H], if given)."""
    torch = _torch()
    _require_cuda(x, Wgu, sgu, Wd, sd, bgu, bd, residual)
    M, H = x.shape
    I = sgu.shape[0] // 2
    _check_residual(residual, M, H)
    y = out if out is not None else torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
    need = workspace_bytes(CK_OP_SWIGLU_MLP, M, H, I, wlayout)
    ws = workspace if workspace is not None else _workspace(need, x.device)
    _check(lib().ck_swiglu_mlp(x.data_ptr(), M, H, I, Wgu.data_ptr(), sgu.data_ptr(), _ptr(bgu),
                               Wd.data_ptr(), sd.data_ptr(), _ptr(bd), _ptr(residual), wlayout, g,
                               y.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream)),
           "ck_swiglu_mlp")
    return y


def gemv_smallM(x, Wpacked, N: int, g: int, bias=None, act: str = "none", out=None,
                workspace=None, stream=None, residual=None, wlayout: int = CK_WLAYOUT_GEMV_PACKED):
    """Small-M (M <= 8) GEMV over a GEMV-resident layout (INT8, or the W6A8 / W4A8
    ones) -> y bf16 [M, N] (+ residual)."""
    torch = _torch()
    _require_cuda(x, Wpacked, bias, residual)
    M, ldx = x.shape
    K = ldx // 2 if act == "swiglu" else ldx
    _check_residual(residual, M, N)
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    need = workspace_bytes(CK_OP_GEMV_SMALLM, M, K, N)
    ws = workspace if workspace is not None else _workspace(need, x.device)
    if wlayout == CK_WLAYOUT_GEMV_PACKED:
        _check(lib().ck_int8_gemv_smallM(x.data_ptr(), M, K, ldx, _ACTS[act], Wpacked.data_ptr(), N,
                                         g, _ptr(bias), _ptr(residual), y.data_ptr(), ws.data_ptr(),
                                         ws.numel(), _stream(stream)), "ck_int8_gemv_smallM")
    else:
        _check(lib().ck_packed_gemv_smallM(x.data_ptr(), M, K, ldx, _ACTS[act], Wpacked.data_ptr(),
                                           wlayout, N, g, _ptr(bias), _ptr(residual), y.data_ptr(),
                                           ws.data_ptr(), ws.numel(), _stream(stream)),
               "ck_packed_gemv_smallM")
    return y


def int8_gemv_dequant(xq, sx, Wpacked, N: int, bias=None, out=None, stream=None, residual=None):
    """Small-M GEMV + dequant on INT8 codes (rotate_quantize_act) and a packed weight -> y bf16 [M, N]."""
    torch = _torch()
    _require_cuda(xq, sx, Wpacked, bias, residual)
    if xq.dtype != torch.int8:
        raise TypeError("int8_gemv_dequant takes the INT8 codes of rotate_quantize_act")
    M, K = xq.shape
    _check_residual(residual, M, N)
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=xq.device)
    _check(lib().ck_int8_gemv_dequant(xq.data_ptr(), sx.data_ptr(), M, K, Wpacked.data_ptr(), N,
                                      _ptr(bias), _ptr(residual), y.data_ptr(), _stream(stream)),
           "ck_int8_gemv_dequant")
    return y


def packed_gemv_dequant(xq, sx, Wpacked, wlayout: int, N: int, bias=None, out=None, stream=None,
                        residual=None):
    """int8_gemv_dequant over any GEMV-resident layout (INT8, W6A8, W4A8) -> y bf16 [M, N]."""
    torch = _torch()
    _require_cuda(xq, sx, Wpacked, bias, residual)
    if xq.dtype != torch.int8:
        raise TypeError("packed_gemv_dequant takes the INT8 codes of rotate_quantize_act")
    M, K = xq.shape
    _check_residual(residual, M, N)
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=xq.device)
    _check(lib().ck_packed_gemv_dequant(xq.data_ptr(), sx.data_ptr(), M, K, Wpacked.data_ptr(),
                                        wlayout, N, _ptr(bias), _ptr(residual), y.data_ptr(),
                                        _stream(stream)), "ck_packed_gemv_dequant")
    return y


def debug_int8_gemm_s32(xq, Wq, stream=None):
    """Raw int32 accumulators of the GEMM engine (test hook)."""
    torch = _torch()
    _require_cuda(xq, Wq)
    M, K = xq.shape
    N = Wq.shape[0]
    acc = torch.empty((M, N), dtype=torch.int32, device=xq.device)
    ws = _workspace(workspace_bytes(CK_OP_DEBUG_GEMM_S32, M, K, N), xq.device)
    _check(lib().ck_debug_int8_gemm_s32(xq.data_ptr(), Wq.data_ptr(), M, N, K, acc.data_ptr(),
                                        ws.data_ptr(), ws.numel(), _stream(stream)),
           "ck_debug_int8_gemm_s32")
    return acc


def debug_gemv_s32(xq, Wpacked, wlayout: int, N: int, stream=None):
    """Exact int32 sums of the small-M GEMV engines on INT8 codes xq [M, K] and a
    GEMV-resident weight (test hook): the weight codes as the engines see them
    on the INT8 grid (6- / 4-bit codes times 4 / 16)."""
    torch = _torch()
    _require_cuda(xq, Wpacked)
    M, K = xq.shape
    acc = torch.empty((M, N), dtype=torch.int32, device=xq.device)
    _check(lib().ck_debug_gemv_s32(xq.data_ptr(), M, K, Wpacked.data_ptr(), wlayout, N,
                                   acc.data_ptr(), _stream(stream)), "ck_debug_gemv_s32")
    return acc


def poll_device_status(stream=None) -> int:
    """Synchronize the stream; CK_OK or CK_ERR_TIMEOUT from the device status word."""
    return int(lib().ck_poll_device_status(_stream(stream)))


def set_wait_timeout_ns(ns: int) -> None:
    lib().ck_set_wait_timeout_ns(int(ns))


def set_launch_overlap(on: bool) -> None:
    """Overlapped launches across calls (ck_set_launch_overlap): the GEMM / GEMV
    may read the weight operands before the work ahead of it on the stream has
    finished, so those weights must be settled (prepared, then synchronized)."""
    lib().ck_set_launch_overlap(1 if on else 0)


def debug_gemm_tile_choice(M: int, N: int, K: int, sms: int) -> int:
    """The GEMM tile code the engine picks for M x K -> N on a GPU of sms SMs (host only)."""
    return int(lib().ck_debug_gemm_tile_choice(int(M), int(N), int(K), int(sms)))


def debug_force_gemm_tile(bn: int) -> None:
    """Force the GEMM tile width (64/128/256); 0 restores the automatic choice."""
    lib().ck_debug_force_gemm_tile(int(bn))


def debug_force_gemv_quantizer(mode: int) -> None:
    """1: quantizer kernel + GEMV, 2: quantize inside the GEMV's CTAs where the
    shape allows; 0 restores the automatic choice."""
    lib().ck_debug_force_gemv_quantizer(int(mode))


def debug_stalled_wait(stream=None) -> int:
    return int(lib().ck_debug_stalled_wait(_stream(stream)))
