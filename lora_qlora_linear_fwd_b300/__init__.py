"""Thin Python binding of the fused LoRA / QLoRA projection library.

Each function here has the name of a C entry point of
``include/lora_b300.h`` and only marshals arguments: shapes come from the
tensors, pointers from ``tensor.data_ptr()``, the stream from torch's current
stream.  All computation runs in the CUDA kernels of
``_lib/liblora_b300.so``; there is no fallback.  Importing the package fails
if the library has not been built (``python
lora_qlora_linear_fwd_b300/build.py``).
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import lib_path

__all__ = [
    "LoraError", "Weight", "dense_weight", "bf16_weight", "nf4_weight", "workspace",
    "workspace_size", "dtype_code",
    "lora_linear_fwd", "lora_linear_bwd", "lora_linear_bwd_noalloc", "lora_linear_fwd_dropout",
    "lora_linear_bwd_dropout", "lora_qk_rope_fwd",
    "lora_qk_rope_bwd", "lora_swiglu_fwd", "lora_swiglu_bwd", "lora_merge",
    "nf4_dequant", "nf4_quantize", "lora_rope_cache_build", "lora_rope_cache_bytes", "lora_nf4_stage_bytes",
    "lora_read_device_status", "lora_clear_device_status", "lora_status_string",
    "lora_kernel_launch_count", "lora_profile_begin", "lora_profile_end",
    "OP_FWD", "OP_BWD", "OP_QK_ROPE_FWD", "OP_QK_ROPE_BWD", "OP_SWIGLU_FWD", "OP_SWIGLU_BWD",
    "OP_MERGE", "OP_MERGE_NF4", "OP_FWD_DROPOUT", "OP_BWD_DROPOUT", "OP_FLAG_DQ", "EXPORTS",
    "library", "DTYPE_BF16", "DTYPE_FP16",
]

OP_FWD, OP_BWD, OP_QK_ROPE_FWD, OP_QK_ROPE_BWD = 0, 1, 2, 3
OP_SWIGLU_FWD, OP_SWIGLU_BWD = 4, 5
OP_MERGE, OP_MERGE_NF4 = 6, 7
OP_FWD_DROPOUT, OP_BWD_DROPOUT = 8, 9
OP_FLAG_DQ = 0x100
WEIGHT_DENSE, WEIGHT_NF4 = 0, 1
DTYPE_BF16, DTYPE_FP16 = 0, 1
STATUS_NAMES = ["LORA_OK", "LORA_ERR_INVALID_ARG", "LORA_ERR_UNSUPPORTED", "LORA_ERR_WORKSPACE",
                "LORA_ERR_ARCH", "LORA_ERR_CUDA", "LORA_ERR_TIMEOUT"]


class LoraError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"{where}: {name}")


class Weight(ctypes.Structure):
    """``lora_weight_t``."""
    _fields_ = [("type", ctypes.c_int), ("w", ctypes.c_void_p), ("absmax", ctypes.c_void_p),
                ("blocksize", ctypes.c_int), ("dtype", ctypes.c_int),
                ("absmax_scale", ctypes.c_void_p), ("absmax_offset", ctypes.c_void_p)]


_P, _I, _F, _D, _Z, _U32P = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double,
                             ctypes.c_size_t, ctypes.POINTER(ctypes.c_uint32))
_U64 = ctypes.c_uint64

# name -> (restype, argtypes); mirrors include/lora_b300.h
EXPORTS = {
    "lora_workspace_size": (_Z, [_I, _I, _I, _I, _I]),
    "lora_linear_fwd": (_I, [_P, Weight, _P, _P, _P, _I, _I, _I, _I, _F, _P, _Z, _P]),
    "lora_linear_bwd": (_I, [_P, Weight, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _F, _P, _Z,
                             _P]),
    "lora_qk_rope_fwd": (_I, [_P, Weight, _P, _P, Weight, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                              _F, _D, _P, _P, _I, _P, _Z, _P]),
    "lora_qk_rope_bwd": (_I, [_P, Weight, _P, _P, Weight, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P,
                              _I, _I, _I, _I, _I, _I, _F, _D, _P, _P, _I, _P, _Z, _P]),
    "lora_swiglu_fwd": (_I, [_P, Weight, _P, _P, Weight, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F,
                             _P, _Z, _P]),
    "lora_swiglu_bwd": (_I, [_P, Weight, _P, _P, Weight, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P,
                             _P, _I, _I, _I, _I, _F, _P, _Z, _P]),
    "lora_linear_bwd_noalloc": (_I, [_P, Weight, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _F,
                                     _P]),
    "lora_linear_fwd_dropout": (_I, [_P, Weight, _P, _P, _P, _I, _I, _I, _I, _F, _F, _U64,
                                     _U64, _P, _Z, _P]),
    "lora_linear_bwd_dropout": (_I, [_P, Weight, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I,
                                     _F, _F, _U64, _U64, _P, _Z, _P]),
    "lora_merge": (_I, [Weight, _P, _P, _I, _I, _I, _F, _I, _P, _Z, _P]),
    "nf4_dequant": (_I, [Weight, _P, _I, _I, _P]),
    "nf4_quantize": (_I, [_P, Weight, _I, _I, _P]),
    "lora_rope_cache_bytes": (_Z, [_I, _I]),
    "lora_nf4_stage_bytes": (_Z, [_I, _I]),
    "lora_rope_cache_build": (_I, [_P, _I, _I, _D, _P]),
    "lora_read_device_status": (_I, [_P, _U32P, _P]),
    "lora_clear_device_status": (_I, [_P, _P]),
    "lora_kernel_launch_count": (ctypes.c_uint64, []),
    "lora_profile_begin": (_I, [_I]),
    "lora_profile_end": (_I, [ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float), _I,
                              ctypes.POINTER(ctypes.c_int)]),
    "lora_status_string": (ctypes.c_char_p, [_I]),
}


def _load():
    path = lib_path()
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python "
                          "lora_qlora_linear_fwd_b300/build.py` (no fallback exists)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in EXPORTS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


library = _load()


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, where: str):
    if status != 0:
        raise LoraError(status, where)


def dtype_code(dtype) -> int:
    """``LORA_DTYPE_*`` of a torch 16-bit floating dtype."""
    if dtype == torch.bfloat16:
        return DTYPE_BF16
    if dtype == torch.float16:
        return DTYPE_FP16
    raise TypeError(f"16-bit type bf16 or fp16 expected, got {dtype}")


def dense_weight(w: torch.Tensor) -> Weight:
    """A dense W [n, k] (bf16 or fp16: the call's 16-bit type)."""
    return Weight(WEIGHT_DENSE, w.data_ptr(), None, 0, dtype_code(w.dtype), None, None)


bf16_weight = dense_weight


def nf4_weight(codes: torch.Tensor, absmax: torch.Tensor, blocksize: int = 64,
               dtype=torch.bfloat16, absmax_scale=None, absmax_offset=None) -> Weight:
    """An NF4 W: codes [n, k/2] and bf16 absmax [n, k/64], or with double
    quantisation uint8 E4M3 absmax codes, fp32 absmax_scale [ceil(n·k/16384)]
    and a one-element fp32 absmax_offset.  ``dtype`` is the call's 16-bit
    type."""
    return Weight(WEIGHT_NF4, codes.data_ptr(), absmax.data_ptr(), blocksize, dtype_code(dtype),
                  None if absmax_scale is None else absmax_scale.data_ptr(),
                  None if absmax_offset is None else absmax_offset.data_ptr())


def _weight(W) -> Weight:
    return W if isinstance(W, Weight) else dense_weight(W)


def workspace_size(op: int, M: int, k: int, n: int, r: int) -> int:
    return int(library.lora_workspace_size(op, M, k, n, r))


def workspace(op: int, M: int, k: int, n: int, r: int, device="cuda", extra: int = 0):
    """A zeroed workspace (status word cleared) of the size the op needs
    (``op`` may carry OP_FLAG_DQ)."""
    nbytes = workspace_size(op, M, k, n, r)
    if nbytes == 0:
        raise LoraError(1, "lora_workspace_size")
    return torch.zeros(nbytes + extra, dtype=torch.uint8, device=device)


def lora_kernel_launch_count() -> int:
    return int(library.lora_kernel_launch_count())


def lora_profile_begin(capacity: int):
    """Open a per-launch timing session for the next ``capacity`` launches."""
    _check(library.lora_profile_begin(int(capacity)), "lora_profile_begin")


def lora_profile_end(capacity: int):
    """Close the session: ``[(kernel_name, ms), ...]`` in launch order."""
    names = (ctypes.c_char_p * capacity)()
    ms = (ctypes.c_float * capacity)()
    count = ctypes.c_int(0)
    _check(library.lora_profile_end(names, ms, int(capacity), ctypes.byref(count)),
           "lora_profile_end")
    return [(names[i].decode(), float(ms[i])) for i in range(count.value)]


def lora_status_string(s: int) -> str:
    return library.lora_status_string(s).decode()


def lora_linear_fwd(x, W, A, B, y, alpha: float, ws, stream=None):
    M, k = x.shape
    n, r = y.shape[1], A.shape[0]
    _check(library.lora_linear_fwd(_ptr(x), _weight(W), _ptr(A), _ptr(B), _ptr(y), M, k, n, r,
                                   float(alpha), _ptr(ws), ws.numel(), _stream(stream)),
           "lora_linear_fwd")


def lora_linear_bwd(x, W, A, B, dy, dx, dA, dB, alpha: float, ws, accumulate_dx: bool = False,
                    stream=None):
    M, k = x.shape
    n, r = dy.shape[1], A.shape[0]
    _check(library.lora_linear_bwd(_ptr(x), _weight(W), _ptr(A), _ptr(B), _ptr(dy), _ptr(dx),
                                   int(bool(accumulate_dx)), _ptr(dA), _ptr(dB), M, k, n, r,
                                   float(alpha), _ptr(ws), ws.numel(), _stream(stream)),
           "lora_linear_bwd")


def lora_linear_bwd_noalloc(x, W, A, B, dy, dx, dA, dB, alpha: float,
                            accumulate_dx: bool = False, stream=None):
    """lora_linear_bwd without a workspace (the library's fixed device
    scratch is used instead; see the C header for its limits)."""
    M, k = x.shape
    n, r = dy.shape[1], A.shape[0]
    _check(library.lora_linear_bwd_noalloc(_ptr(x), _weight(W), _ptr(A), _ptr(B), _ptr(dy),
                                           _ptr(dx), int(bool(accumulate_dx)), _ptr(dA),
                                           _ptr(dB), M, k, n, r, float(alpha), _stream(stream)),
           "lora_linear_bwd_noalloc")


def lora_qk_rope_fwd(x, Wq, Aq, Bq, Wk, Ak, Bk, q, k_out, alpha: float, rope_theta: float,
                     positions, cos_sin_cache, max_pos: int, ws, head_dim: int = 128,
                     stream=None):
    M, hidden = x.shape
    r = Aq.shape[0]
    _check(library.lora_qk_rope_fwd(
        _ptr(x), _weight(Wq), _ptr(Aq), _ptr(Bq), _weight(Wk), _ptr(Ak), _ptr(Bk), _ptr(q),
        _ptr(k_out), M, hidden, q.shape[1] // head_dim, k_out.shape[1] // head_dim, head_dim, r,
        float(alpha), float(rope_theta), _ptr(positions), _ptr(cos_sin_cache), int(max_pos),
        _ptr(ws), ws.numel(), _stream(stream)), "lora_qk_rope_fwd")


def lora_qk_rope_bwd(x, Wq, Aq, Bq, Wk, Ak, Bk, dq, dk, dx, dAq, dBq, dAk, dBk, alpha: float,
                     rope_theta: float, positions, cos_sin_cache, max_pos: int, ws,
                     head_dim: int = 128, accumulate_dx: bool = False, stream=None):
    M, hidden = x.shape
    r = Aq.shape[0]
    _check(library.lora_qk_rope_bwd(
        _ptr(x), _weight(Wq), _ptr(Aq), _ptr(Bq), _weight(Wk), _ptr(Ak), _ptr(Bk), _ptr(dq),
        _ptr(dk), _ptr(dx), int(bool(accumulate_dx)), _ptr(dAq), _ptr(dBq), _ptr(dAk),
        _ptr(dBk), M, hidden, dq.shape[1] // head_dim, dk.shape[1] // head_dim, head_dim, r,
        float(alpha), float(rope_theta), _ptr(positions), _ptr(cos_sin_cache), int(max_pos),
        _ptr(ws), ws.numel(), _stream(stream)), "lora_qk_rope_bwd")


def lora_swiglu_fwd(x, Wg, Ag, Bg, Wu, Au, Bu, h, alpha: float, ws, g=None, u=None,
                    stream=None):
    """h = silu(g)·u of the gate and up LoRA projections; g and u are also
    written when given (the backward needs them)."""
    M, k = x.shape
    n, r = h.shape[1], Ag.shape[0]
    _check(library.lora_swiglu_fwd(_ptr(x), _weight(Wg), _ptr(Ag), _ptr(Bg), _weight(Wu),
                                   _ptr(Au), _ptr(Bu), _ptr(h), _ptr(g), _ptr(u), M, k, n, r,
                                   float(alpha), _ptr(ws), ws.numel(), _stream(stream)),
           "lora_swiglu_fwd")


def lora_swiglu_bwd(x, Wg, Ag, Bg, Wu, Au, Bu, g, u, dh, dx, dAg, dBg, dAu, dBu, alpha: float,
                    ws, accumulate_dx: bool = False, stream=None):
    M, k = x.shape
    n, r = dh.shape[1], Ag.shape[0]
    _check(library.lora_swiglu_bwd(_ptr(x), _weight(Wg), _ptr(Ag), _ptr(Bg), _weight(Wu),
                                   _ptr(Au), _ptr(Bu), _ptr(g), _ptr(u), _ptr(dh), _ptr(dx),
                                   int(bool(accumulate_dx)), _ptr(dAg), _ptr(dBg), _ptr(dAu),
                                   _ptr(dBu), M, k, n, r, float(alpha), _ptr(ws), ws.numel(),
                                   _stream(stream)), "lora_swiglu_bwd")


def lora_linear_fwd_dropout(x, W, A, B, y, alpha: float, dropout_p: float, seed: int,
                            offset: int, ws, stream=None):
    M, k = x.shape
    n, r = y.shape[1], A.shape[0]
    _check(library.lora_linear_fwd_dropout(_ptr(x), _weight(W), _ptr(A), _ptr(B), _ptr(y), M, k,
                                           n, r, float(alpha), float(dropout_p), int(seed),
                                           int(offset), _ptr(ws), ws.numel(), _stream(stream)),
           "lora_linear_fwd_dropout")


def lora_linear_bwd_dropout(x, W, A, B, dy, dx, dA, dB, alpha: float, dropout_p: float,
                            seed: int, offset: int, ws, accumulate_dx: bool = False,
                            stream=None):
    M, k = x.shape
    n, r = dy.shape[1], A.shape[0]
    _check(library.lora_linear_bwd_dropout(_ptr(x), _weight(W), _ptr(A), _ptr(B), _ptr(dy),
                                           _ptr(dx), int(bool(accumulate_dx)), _ptr(dA),
                                           _ptr(dB), M, k, n, r, float(alpha), float(dropout_p),
                                           int(seed), int(offset), _ptr(ws), ws.numel(),
                                           _stream(stream)), "lora_linear_bwd_dropout")


def lora_merge(W, A, B, alpha: float, sign: int = 1, ws=None, stream=None):
    """W <- W + sign·(alpha/r)·B·A in place: a dense W tensor [n, k], or an
    NF4 ``Weight`` (dequantised, merged and re-quantised in place)."""
    n, r = B.shape
    k = A.shape[1]
    Wd = _weight(W)
    op = OP_MERGE_NF4 if Wd.type == WEIGHT_NF4 else OP_MERGE
    if ws is None:
        ws = workspace(op, 1, k, n, r, device=A.device)
    _check(library.lora_merge(Wd, _ptr(A), _ptr(B), n, k, r, float(alpha), int(sign), _ptr(ws),
                              ws.numel(), _stream(stream)), "lora_merge")


def nf4_dequant(W: Weight, w_out, stream=None):
    """w_out [n, k] (the weight's 16-bit type) from an NF4 ``Weight``."""
    n, k = w_out.shape
    _check(library.nf4_dequant(W, _ptr(w_out), n, k, _stream(stream)), "nf4_dequant")


def nf4_quantize(w, W_out: Weight, stream=None):
    """Quantise a 16-bit w [n, k] into the codes and block scales W_out
    points at (double-quantised when W_out has absmax_scale)."""
    n, k = w.shape
    _check(library.nf4_quantize(_ptr(w), W_out, n, k, _stream(stream)), "nf4_quantize")


def lora_nf4_stage_bytes(n: int, k: int) -> int:
    """Workspace bytes that let an NF4 call stage W [n, k] in 16-bit."""
    return int(library.lora_nf4_stage_bytes(int(n), int(k)))


def lora_rope_cache_bytes(max_pos: int, head_dim: int = 128) -> int:
    return int(library.lora_rope_cache_bytes(max_pos, head_dim))


def lora_rope_cache_build(cos_sin, max_pos: int, head_dim: int, theta: float, stream=None):
    _check(library.lora_rope_cache_build(_ptr(cos_sin), int(max_pos), int(head_dim),
                                         float(theta), _stream(stream)), "lora_rope_cache_build")


def lora_read_device_status(ws, stream=None) -> int:
    out = ctypes.c_uint32(0)
    s = library.lora_read_device_status(_ptr(ws), ctypes.byref(out), _stream(stream))
    if s not in (0, 6):
        raise LoraError(s, "lora_read_device_status")
    return int(out.value)


def lora_clear_device_status(ws, stream=None):
    _check(library.lora_clear_device_status(_ptr(ws), _stream(stream)), "lora_clear_device_status")
