"""Thin ctypes binding of the C ABI in ``include/qlora.h``.

Argument marshalling only: every step of the QLoRA hot path runs in the CUDA
kernels of ``libqlora_b300.so``.  PyTorch supplies device memory and the
current stream.  There is no fallback: if the library is missing, or a call
returns an error status, the binding raises.

The function names follow the C ABI:
  qlora_nf4_sizes, qlora_quantize_nf4, qlora_dequant, qlora_merge_lora, qlora_workspace_size,
  qlora_workspace_size_min, qlora_workspace_init, qlora_device_status, qlora_linear_fwd,
  qlora_linear_bwd, qlora_nf4_thresholds, qlora_nf4_codebook.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqlora_b300.so")

QLORA_OK = 0
QLORA_ERR_TIMEOUT = 6
QLORA_F32, QLORA_BF16 = 0, 1
QLORA_FLAG_FORCE_GEMV, QLORA_FLAG_FORCE_GEMM = 1, 2

# Every symbol the header declares (checked by the CPU tests).
EXPORTED = (
    "qlora_nf4_sizes", "qlora_quantize_nf4", "qlora_dequant", "qlora_workspace_size",
    "qlora_workspace_init", "qlora_device_status", "qlora_linear_fwd", "qlora_linear_bwd",
    "qlora_nf4_thresholds", "qlora_nf4_codebook", "qlora_status_string",
    "qlora_linear_bwd_noalloc", "qlora_workspace_size_min", "qlora_merge_lora",
    "qlora_dropout_mask_words", "qlora_dropout_mask", "qlora_linear_fwd_dropout",
    "qlora_linear_bwd_dropout",
)


class QloraError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: status {status} ({msg})")
        self.status = status


class _DropoutStruct(ctypes.Structure):
    _fields_ = [("mask", ctypes.c_void_p), ("p", ctypes.c_float)]


class _NF4WeightStruct(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("block", ctypes.c_int32),
                ("group", ctypes.c_int32), ("codebook", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("packed", ctypes.c_void_p),
                ("absmax_code", ctypes.c_void_p), ("absmax_f32", ctypes.c_void_p),
                ("scale2", ctypes.c_void_p)]


_lib = None


def load(path: str = LIB_PATH):
    """Load the shared library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: run `python -m bit_nf4_quantized_35_b300.build`")
    lib = ctypes.CDLL(path)
    P, i64, i32, u32, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32,
                            ctypes.c_size_t)
    f32 = ctypes.c_float
    st = ctypes.c_int
    sig = {
        "qlora_nf4_sizes": [i64, i64, i32, i32, P, P, P],
        "qlora_quantize_nf4": [P, st, P, P, P],
        "qlora_dequant": [P, P, P],
        "qlora_merge_lora": [P, P, P, i32, f32, P, P],
        "qlora_dropout_mask_words": [i64, P],
        "qlora_dropout_mask": [ctypes.c_uint64, f32, i64, i64, P, P],
        "qlora_linear_fwd_dropout": [P, P, i64, P, P, i32, f32, P, P, st, P, P, sz, u32, P],
        "qlora_linear_bwd_dropout": [P, P, P, i64, P, P, i32, f32, P, P, P, P, P, P, sz, u32, P],
        "qlora_workspace_size": [i64, i64, i64, i32, P],
        "qlora_workspace_size_min": [i64, i64, i64, i32, P],
        "qlora_workspace_init": [P, sz, P],
        "qlora_device_status": [P, P, P],
        "qlora_linear_fwd": [P, P, i64, P, P, i32, f32, P, st, P, P, sz, u32, P],
        "qlora_linear_bwd": [P, P, P, i64, P, P, i32, f32, P, P, st, P, P, P, sz, u32, P],
        "qlora_linear_bwd_noalloc": [P, P, P, i64, P, P, i32, f32, P, P, st, P, P, u32, P],
        "qlora_nf4_thresholds": [i32, P],
        "qlora_nf4_codebook": [i32, P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = st
    lib.qlora_status_string.argtypes = [st]
    lib.qlora_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(fn: str, status: int):
    if status != QLORA_OK:
        msg = load().qlora_status_string(status).decode()
        raise QloraError(fn, status, msg)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream: torch.cuda.Stream | None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


# ------------------------------------------------------------------ host-only
def nf4_sizes(rows: int, cols: int, block: int = 64, group: int = 256):
    p, c, s = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check("qlora_nf4_sizes", load().qlora_nf4_sizes(rows, cols, block, group, ctypes.byref(p),
                                                      ctypes.byref(c), ctypes.byref(s)))
    return p.value, c.value, s.value


QLORA_CODEBOOK_PRINTED, QLORA_CODEBOOK_QUANTILE = 0, 1


def nf4_thresholds(codebook: int = QLORA_CODEBOOK_PRINTED) -> list[float]:
    out = (ctypes.c_float * 15)()
    _check("qlora_nf4_thresholds", load().qlora_nf4_thresholds(codebook, out))
    return list(out)


def nf4_codebook(codebook: int = QLORA_CODEBOOK_PRINTED) -> list[float]:
    out = (ctypes.c_float * 16)()
    _check("qlora_nf4_codebook", load().qlora_nf4_codebook(codebook, out))
    return list(out)


def workspace_size(M: int, N: int, K: int, r: int) -> int:
    b = ctypes.c_size_t()
    _check("qlora_workspace_size", load().qlora_workspace_size(M, N, K, r, ctypes.byref(b)))
    return b.value


def workspace_size_min(M: int, N: int, K: int, r: int) -> int:
    b = ctypes.c_size_t()
    _check("qlora_workspace_size_min",
           load().qlora_workspace_size_min(M, N, K, r, ctypes.byref(b)))
    return b.value


# ---------------------------------------------------------------- device side
@dataclass
class NF4Weight:
    """Device buffers of one quantised weight (all caller-owned torch tensors)."""
    rows: int
    cols: int
    packed: torch.Tensor               # uint8 [rows*cols/2]
    absmax_code: torch.Tensor | None   # int8 [nblocks]       (group > 0)
    scale2: torch.Tensor | None        # float32 [ngroups]    (group > 0)
    absmax_f32: torch.Tensor | None    # float32 [nblocks]    (group == 0)
    block: int = 64
    group: int = 256
    codebook: int = 0  # qlora_codebook: 0 printed table, 1 quantile formula

    def struct(self) -> _NF4WeightStruct:
        return _NF4WeightStruct(self.rows, self.cols, self.block, self.group, self.codebook, 0,
                                self.packed.data_ptr(),
                                None if self.absmax_code is None else self.absmax_code.data_ptr(),
                                None if self.absmax_f32 is None else self.absmax_f32.data_ptr(),
                                None if self.scale2 is None else self.scale2.data_ptr())

    @staticmethod
    def empty(rows: int, cols: int, device="cuda", block: int = 64, group: int = 256,
              codebook: int = 0):
        pb, cb, sb = nf4_sizes(rows, cols, block, group)
        packed = torch.empty(max(pb, 16), dtype=torch.uint8, device=device)[:pb]
        if group > 0:
            codes = torch.empty(max(cb, 16), dtype=torch.int8, device=device)[:cb]
            s2 = torch.empty(max(sb // 4, 4), dtype=torch.float32, device=device)[:sb // 4]
            return NF4Weight(rows, cols, packed, codes, s2, None, block, group, codebook)
        absf = torch.empty(max(cb // 4, 4), dtype=torch.float32, device=device)[:cb // 4]
        return NF4Weight(rows, cols, packed, None, None, absf, block, group, codebook)


def quantize_nf4(W: torch.Tensor, group: int = 256, out: NF4Weight | None = None,
                 nonfinite_flag: torch.Tensor | None = None, stream=None,
                 block: int = 64, codebook: int = 0) -> NF4Weight:
    """qlora_quantize_nf4 on a contiguous fp32 or bf16 CUDA matrix [rows, cols]."""
    assert W.is_cuda and W.is_contiguous() and W.dim() == 2
    dt = {torch.float32: QLORA_F32, torch.bfloat16: QLORA_BF16}[W.dtype]
    rows, cols = W.shape
    if out is None:
        out = NF4Weight.empty(rows, cols, W.device, block=block, group=group,
                              codebook=codebook)
    s = out.struct()
    _check("qlora_quantize_nf4", load().qlora_quantize_nf4(
        _ptr(W), dt, ctypes.byref(s), _ptr(nonfinite_flag), _stream(stream)))
    return out


def dequant(w: NF4Weight, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """qlora_dequant -> bf16 [rows, cols]."""
    if out is None:
        out = torch.empty((w.rows, w.cols), dtype=torch.bfloat16, device=w.packed.device)
    s = w.struct()
    _check("qlora_dequant", load().qlora_dequant(ctypes.byref(s), _ptr(out), _stream(stream)))
    return out


def merge_lora(w: NF4Weight, A: torch.Tensor, B: torch.Tensor, alpha: float,
               out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """qlora_merge_lora -> bf16 [rows, cols] = bf16(W_hat + alpha/r B A)."""
    r = A.shape[0]
    if out is None:
        out = torch.empty((w.rows, w.cols), dtype=torch.bfloat16, device=w.packed.device)
    s = w.struct()
    _check("qlora_merge_lora", load().qlora_merge_lora(
        ctypes.byref(s), _ptr(A), _ptr(B), r, float(alpha), _ptr(out), _stream(stream)))
    return out


class Workspace:
    """A zero-initialised device workspace sized for (M, N, K, r).

    ``minimal=True`` sizes it with qlora_workspace_size_min (no split-tile
    area: the fused GEMM then computes whole output tiles only)."""

    def __init__(self, M: int, N: int, K: int, r: int, device="cuda", stream=None,
                 minimal: bool = False):
        self.nbytes = (workspace_size_min if minimal else workspace_size)(M, N, K, r)
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        _check("qlora_workspace_init", load().qlora_workspace_init(
            _ptr(self.buf), self.nbytes, _stream(stream)))

    def device_status(self, stream=None) -> int:
        v = ctypes.c_int32()
        _check("qlora_device_status", load().qlora_device_status(
            _ptr(self.buf), ctypes.byref(v), _stream(stream)))
        return v.value


def dropout_mask_words(K: int) -> int:
    v = ctypes.c_int64()
    _check("qlora_dropout_mask_words", load().qlora_dropout_mask_words(K, ctypes.byref(v)))
    return v.value


def dropout_mask(seed: int, p: float, M: int, K: int, device="cuda", out=None,
                 stream=None) -> torch.Tensor:
    """qlora_dropout_mask -> int32 tensor [M, words_per_row] of keep bits."""
    if out is None:
        out = torch.empty((M, dropout_mask_words(K)), dtype=torch.int32, device=device)
    _check("qlora_dropout_mask", load().qlora_dropout_mask(
        ctypes.c_uint64(seed), float(p), M, K, _ptr(out), _stream(stream)))
    return out


def linear_fwd(w: NF4Weight, x: torch.Tensor, A: torch.Tensor, B: torch.Tensor, alpha: float,
               ws: Workspace, y: torch.Tensor | None = None, y_dtype=torch.float32,
               t_save: torch.Tensor | None = None, flags: int = 0, stream=None,
               dropout: tuple | None = None) -> torch.Tensor:
    """qlora_linear_fwd: y = x W_hat^T + (x A^T) B^T alpha/r; with
    dropout=(mask, p) qlora_linear_fwd_dropout."""
    M = x.shape[0]
    r = A.shape[0]
    if y is None:
        y = torch.empty((M, w.rows), dtype=y_dtype, device=x.device)
    ydt = {torch.float32: QLORA_F32, torch.bfloat16: QLORA_BF16}[y.dtype]
    s = w.struct()
    if dropout is not None:
        d = _DropoutStruct(dropout[0].data_ptr(), float(dropout[1]))
        _check("qlora_linear_fwd_dropout", load().qlora_linear_fwd_dropout(
            ctypes.byref(s), _ptr(x), M, _ptr(A), _ptr(B), r, float(alpha), ctypes.byref(d),
            _ptr(y), ydt, _ptr(t_save), _ptr(ws.buf), ws.nbytes, flags, _stream(stream)))
        return y
    _check("qlora_linear_fwd", load().qlora_linear_fwd(
        ctypes.byref(s), _ptr(x), M, _ptr(A), _ptr(B), r, float(alpha), _ptr(y), ydt,
        _ptr(t_save), _ptr(ws.buf), ws.nbytes, flags, _stream(stream)))
    return y


def linear_bwd_noalloc(w: NF4Weight, x: torch.Tensor, dY: torch.Tensor, A: torch.Tensor,
                       B: torch.Tensor, alpha: float, t_saved: torch.Tensor | None = None,
                       dX: torch.Tensor | None = None, dx_dtype=torch.float32,
                       dA: torch.Tensor | None = None, dB: torch.Tensor | None = None,
                       flags: int = 0, stream=None):
    """qlora_linear_bwd_noalloc -> (dX, dA, dB): the backward without a
    caller workspace (the library's fixed device scratch array is used)."""
    M = x.shape[0]
    r = A.shape[0]
    dev = x.device
    if dX is None:
        dX = torch.empty((M, w.cols), dtype=dx_dtype, device=dev)
    if dA is None:
        dA = torch.empty((r, w.cols), dtype=torch.float32, device=dev)
    if dB is None:
        dB = torch.empty((w.rows, r), dtype=torch.float32, device=dev)
    dxt = {torch.float32: QLORA_F32, torch.bfloat16: QLORA_BF16}[dX.dtype]
    s = w.struct()
    _check("qlora_linear_bwd_noalloc", load().qlora_linear_bwd_noalloc(
        ctypes.byref(s), _ptr(x), _ptr(dY), M, _ptr(A), _ptr(B), r, float(alpha),
        _ptr(t_saved), _ptr(dX), dxt, _ptr(dA), _ptr(dB), flags, _stream(stream)))
    return dX, dA, dB


def linear_bwd(w: NF4Weight, x: torch.Tensor, dY: torch.Tensor, A: torch.Tensor,
               B: torch.Tensor, alpha: float, ws: Workspace, t_saved: torch.Tensor | None = None,
               dX: torch.Tensor | None = None, dx_dtype=torch.float32,
               dA: torch.Tensor | None = None, dB: torch.Tensor | None = None, flags: int = 0,
               stream=None, dropout: tuple | None = None):
    """qlora_linear_bwd -> (dX, dA, dB); with dropout=(mask, p)
    qlora_linear_bwd_dropout (fp32 dX)."""
    M = x.shape[0]
    r = A.shape[0]
    dev = x.device
    if dX is None:
        dX = torch.empty((M, w.cols), dtype=dx_dtype, device=dev)
    if dA is None:
        dA = torch.empty((r, w.cols), dtype=torch.float32, device=dev)
    if dB is None:
        dB = torch.empty((w.rows, r), dtype=torch.float32, device=dev)
    dxt = {torch.float32: QLORA_F32, torch.bfloat16: QLORA_BF16}[dX.dtype]
    s = w.struct()
    if dropout is not None:
        d = _DropoutStruct(dropout[0].data_ptr(), float(dropout[1]))
        _check("qlora_linear_bwd_dropout", load().qlora_linear_bwd_dropout(
            ctypes.byref(s), _ptr(x), _ptr(dY), M, _ptr(A), _ptr(B), r, float(alpha),
            ctypes.byref(d), _ptr(t_saved), _ptr(dX), _ptr(dA), _ptr(dB), _ptr(ws.buf),
            ws.nbytes, flags, _stream(stream)))
        return dX, dA, dB
    _check("qlora_linear_bwd", load().qlora_linear_bwd(
        ctypes.byref(s), _ptr(x), _ptr(dY), M, _ptr(A), _ptr(B), r, float(alpha),
        _ptr(t_saved), _ptr(dX), dxt, _ptr(dA), _ptr(dB), _ptr(ws.buf), ws.nbytes, flags,
        _stream(stream)))
    return dX, dA, dB
