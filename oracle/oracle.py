"""CPU oracle for the QLoRA NF4 hot path -- Python side (ctypes over numpy).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module.  The product
library never imports, links or executes anything under ``oracle/``, and the
oracle never imports the product package: the two share nothing but the
seeded input generators (``bit_nf4_quantized_35_b300/inputs.py``), which hold
none of the method's arithmetic.

The arithmetic lives in ``qlora_oracle.c`` (plain C, binary32 decisions,
binary64 contractions).  Each wrapper below names the C function it calls and
the passage that function follows; see the C file's header for the pages.

Parity status: every function is pinned by ``tests/test_oracle_*.py``.  The
three conventions the pages leave open -- the double-quantisation layout and
rounding, the nibble order, and the tie-break -- are pinned only by the
conventions stated in the C source ("parity unpinned" by the pages).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qlora_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

# binary32 semantics: no contraction into FMA, no fast math, SSE arithmetic.
CFLAGS = ["-O2", "-fPIC", "-shared", "-std=c11", "-fopenmp", "-ffp-contract=off",
          "-fno-fast-math", "-fexcess-precision=standard", "-Wall"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``qlora_oracle.c`` (or another copy of it) into a shared library."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def _declare(lib):
    P = ctypes.c_void_p
    i64, i32, u32, f64 = ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32, ctypes.c_double
    lib.oracle_nf4_codebook.argtypes = [P]
    lib.oracle_nf4_codebook.restype = None
    lib.oracle_nearest_code.argtypes = [ctypes.c_float]
    lib.oracle_nearest_code.restype = ctypes.c_int
    lib.oracle_nearest_codes_bits.argtypes = [u32, i64, P]
    lib.oracle_nearest_codes_bits.restype = None
    lib.oracle_nearest_codes_scaled_bits.argtypes = [u32, i64, ctypes.c_float, P]
    lib.oracle_nearest_codes_scaled_bits.restype = None
    lib.oracle_bf16_rne_array.argtypes = [P, i64, P]
    lib.oracle_bf16_rne_array.restype = None
    lib.oracle_quantize_nf4.argtypes = [P, i64, i64, i32, i32, P, P, P, P, P, i32]
    lib.oracle_quantize_nf4.restype = i64
    lib.oracle_dequant_bf16.argtypes = [P, P, P, P, i64, i64, i32, i32, P, i32]
    lib.oracle_codebook_values.argtypes = [i32, P]
    lib.oracle_codebook_values.restype = None
    lib.oracle_inv_normal.argtypes = [f64]
    lib.oracle_inv_normal.restype = f64
    lib.oracle_nearest_code_cb.argtypes = [i32, ctypes.c_float]
    lib.oracle_nearest_code_cb.restype = ctypes.c_int
    lib.oracle_dequant_bf16.restype = ctypes.c_int
    lib.oracle_linear_fwd.argtypes = [P, i64, i64, P, i64, P, P, i32, f64, P, i64, P, P, P, f64]
    lib.oracle_linear_fwd.restype = None
    lib.oracle_linear_bwd.argtypes = [P, P, i64, i64, i64, P, P, P, i32, f64, P, i64,
                                      P, P, P, P, P, P, f64]
    lib.oracle_philox_stream.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
    lib.oracle_philox_stream.restype = ctypes.c_uint64
    lib.oracle_dropout_keep.argtypes = [ctypes.c_uint64, f64, i64, i64, P]
    lib.oracle_dropout_keep.restype = None
    lib.oracle_linear_bwd.restype = None
    lib.oracle_bf16_rne_double.argtypes = [f64]
    lib.oracle_bf16_rne_double.restype = ctypes.c_uint16
    lib.oracle_merge_bf16.argtypes = [P, i64, i64, P, P, i32, f64, P, P]
    lib.oracle_merge_bf16.restype = None
    lib.oracle_nf4_storage_bytes.argtypes = [i64, i64, i32, i32, P, P, P]
    lib.oracle_nf4_storage_bytes.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    lib.oracle_set_num_threads.restype = None
    return lib


def use_library(path: str | None):
    """Point every wrapper of this module at another build of the oracle
    (``None`` restores the default build).  Used by the mutation tests, which
    plant a mistake in a copy of the C source and check that a pin fails."""
    global _lib
    with _lock:
        _lib = None if path is None else _declare(ctypes.CDLL(path))


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
        return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    """Thread count of the oracle's OpenMP loops (results do not depend on it)."""
    _load().oracle_set_num_threads(int(n))


def codebook(which: int = 0) -> np.ndarray:
    """The 16 codepoints as binary32: 0 the printed NF4 table
    (oracle_nf4_codebook), 1 the quantile-formula table."""
    out = np.zeros(16, dtype=np.float32)
    if which == 0:
        _load().oracle_nf4_codebook(_ptr(out))
    else:
        _load().oracle_codebook_values(which, _ptr(out))
    return out


def inv_normal(p: float) -> float:
    """Phi^-1(p) by bisection on the normal CDF (binary64)."""
    return float(_load().oracle_inv_normal(float(p)))


def nearest_code_cb(which: int, xn: float) -> int:
    return int(_load().oracle_nearest_code_cb(which, ctypes.c_float(float(xn))))


def nearest_code(xn: float) -> int:
    """Index of the nearest codepoint of one normalised value."""
    return int(_load().oracle_nearest_code(ctypes.c_float(float(xn))))


def nearest_codes_bits(start_bits: int, count: int) -> np.ndarray:
    """Indices for ``count`` consecutive binary32 bit patterns."""
    out = np.empty(count, dtype=np.uint8)
    _load().oracle_nearest_codes_bits(ctypes.c_uint32(start_bits), count, _ptr(out))
    return out


def nearest_codes_scaled_bits(start_bits: int, count: int, absmax: float) -> np.ndarray:
    """Indices of ``count`` consecutive binary32 weights in a block whose
    absolute maximum is ``absmax`` (division, then nearest codepoint)."""
    out = np.empty(count, dtype=np.uint8)
    _load().oracle_nearest_codes_scaled_bits(ctypes.c_uint32(start_bits), count,
                                             ctypes.c_float(absmax), _ptr(out))
    return out


def bf16_rne(values) -> np.ndarray:
    """binary32 -> bf16 bit patterns (uint16), round to nearest even."""
    v = _f32(values).ravel()
    out = np.empty(v.size, dtype=np.uint16)
    _load().oracle_bf16_rne_array(_ptr(v), v.size, _ptr(out))
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to binary32 values (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


class NF4Weight:
    """Quantised weight as the oracle stores it (numpy arrays)."""

    def __init__(self, rows, cols, block, group, packed, absmax_code, absmax_f32, scale2,
                 idx, nonfinite, codebook=0):
        self.rows, self.cols, self.block, self.group = rows, cols, block, group
        self.codebook = codebook
        self.packed, self.absmax_code, self.absmax_f32, self.scale2 = (
            packed, absmax_code, absmax_f32, scale2)
        self.idx = idx
        self.nonfinite = nonfinite

    @property
    def nblocks(self) -> int:
        return self.rows * self.cols // self.block


def quantize_nf4(w, block: int = 64, group: int = 256, want_idx: bool = True,
                 codebook: int = 0) -> NF4Weight:
    """Blockwise NF4 quantisation (+ double quantisation when group > 0).

    ``w`` is a 2-D array of binary32 values (bf16 inputs widened exactly);
    ``codebook`` 0 is the printed table, 1 the quantile-formula table."""
    w = _f32(w)
    if w.ndim != 2:
        raise ValueError("w must be 2-D [rows, cols]")
    rows, cols = w.shape
    if block <= 0 or block % 2 or cols % block:
        raise ValueError("cols must be a multiple of an even block size")
    n = rows * cols
    nblocks = n // block
    packed = np.zeros(n // 2, dtype=np.uint8)
    codes = np.zeros(nblocks if group > 0 else 0, dtype=np.int8)
    absf = np.zeros(nblocks if group == 0 else 0, dtype=np.float32)
    ngroups = (nblocks + group - 1) // group if group > 0 else 0
    s2 = np.zeros(ngroups, dtype=np.float32)
    idx = np.zeros(n, dtype=np.uint8) if want_idx else None
    nz = lambda a: _ptr(a) if a.size else ctypes.c_void_p(0)
    nonfinite = _load().oracle_quantize_nf4(
        _ptr(w), rows, cols, block, group, _ptr(packed), nz(codes), nz(absf), nz(s2),
        _ptr(idx) if idx is not None else ctypes.c_void_p(0), codebook)
    if nonfinite < 0:
        raise ValueError("oracle_quantize_nf4 rejected its arguments")
    return NF4Weight(rows, cols, block, group, packed, codes, absf, s2,
                     idx.reshape(rows, cols) if idx is not None else None, int(nonfinite),
                     codebook)


def dequant_bf16(q: NF4Weight) -> np.ndarray:
    """Dequantised weight as bf16 bit patterns, shape [rows, cols]."""
    out = np.empty(q.rows * q.cols, dtype=np.uint16)
    nz = lambda a: _ptr(a) if a.size else ctypes.c_void_p(0)
    rc = _load().oracle_dequant_bf16(_ptr(q.packed), nz(q.absmax_code), nz(q.absmax_f32),
                                     nz(q.scale2), q.rows, q.cols, q.block, q.group, _ptr(out),
                                     q.codebook)
    if rc != 0:
        raise ValueError("oracle_dequant_bf16 rejected its arguments")
    return out.reshape(q.rows, q.cols)


def dequant_f32(q: NF4Weight) -> np.ndarray:
    return bf16_bits_to_f32(dequant_bf16(q)).reshape(q.rows, q.cols)


def philox_stream(seed: int, o: int) -> int:
    """The o-th 64-bit output of the Philox4x64-10 stream keyed by seed."""
    return int(_load().oracle_philox_stream(seed, o))


def dropout_keep(seed: int, p: float, M: int, K: int) -> np.ndarray:
    """LoRA dropout keep mask [M, K] (uint8 0/1) for probability p."""
    keep = np.empty((M, K), dtype=np.uint8)
    _load().oracle_dropout_keep(seed, float(p), M, K, _ptr(keep))
    return keep


def _keep_args(keep, p):
    if keep is None:
        return ctypes.c_void_p(0), 1.0, None
    k = np.ascontiguousarray(keep, dtype=np.uint8)
    return _ptr(k), 1.0 / (1.0 - float(p)), k


def linear_fwd(x, w, A, B, alpha: float, rows=None, keep=None, p: float = 0.0):
    """fp64 forward y = x W^T + (x A^T) B^T alpha/r on the listed rows; with
    `keep` ([M, K] 0/1) the LoRA branch takes dropout(x) = x keep / (1 - p).

    Returns (y [nrows, N] float64, t [nrows, r] float64)."""
    x, w, A, B = _f32(x), _f32(w), _f32(A), _f32(B)
    M, K = x.shape
    N = w.shape[0]
    r = A.shape[0]
    assert w.shape == (N, K) and A.shape == (r, K) and B.shape == (N, r)
    rows = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    y = np.zeros((rows.size, N), dtype=np.float64)
    t = np.zeros((rows.size, r), dtype=np.float64)
    kp, ks, _hold = _keep_args(keep, p)
    _load().oracle_linear_fwd(_ptr(x), M, K, _ptr(w), N, _ptr(A), _ptr(B), r, float(alpha),
                              _ptr(rows), rows.size, _ptr(y), _ptr(t), kp, ks)
    return y, t


def linear_bwd(x, dY, w, A, B, alpha: float, rows=None, keep=None, p: float = 0.0):
    """fp64 backward.  Returns dict with dX [nrows, K], dA [r, K], dB [N, r],
    t [M, r], u [M, r] (all float64)."""
    x, dY, w, A, B = _f32(x), _f32(dY), _f32(w), _f32(A), _f32(B)
    M, K = x.shape
    N = w.shape[0]
    r = A.shape[0]
    assert dY.shape == (M, N) and w.shape == (N, K) and A.shape == (r, K) and B.shape == (N, r)
    rows = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    dX = np.zeros((rows.size, K), dtype=np.float64)
    dA = np.zeros((r, K), dtype=np.float64)
    dB = np.zeros((N, r), dtype=np.float64)
    t = np.zeros((M, r), dtype=np.float64)
    u = np.zeros((M, r), dtype=np.float64)
    kp, ks, _hold = _keep_args(keep, p)
    _load().oracle_linear_bwd(_ptr(x), _ptr(dY), M, K, N, _ptr(w), _ptr(A), _ptr(B), r,
                              float(alpha), _ptr(rows), rows.size, _ptr(dX), _ptr(dA),
                              _ptr(dB), _ptr(t), _ptr(u), kp, ks)
    return {"dX": dX, "dA": dA, "dB": dB, "t": t, "u": u}


def bf16_rne_double(v: float) -> int:
    """binary64 -> bf16 bit pattern, round to nearest even (one rounding)."""
    return int(_load().oracle_bf16_rne_double(float(v)))


def merge_bf16(w, A, B, alpha: float):
    """Merged weight W_hat + alpha/r B A: (bf16 bit patterns [N, K] uint16,
    binary64 values before rounding [N, K])."""
    w, A, B = _f32(w), _f32(A), _f32(B)
    N, K = w.shape
    r = A.shape[0]
    assert A.shape == (r, K) and B.shape == (N, r)
    exact = np.empty((N, K), dtype=np.float64)
    bits = np.empty((N, K), dtype=np.uint16)
    _load().oracle_merge_bf16(_ptr(w), N, K, _ptr(A), _ptr(B), r, float(alpha), _ptr(exact),
                              _ptr(bits))
    return bits, exact


def storage_bytes(rows: int, cols: int, block: int = 64, group: int = 256):
    """(packed, constants, second-level scales) byte counts for one matrix."""
    p, c, s = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    rc = _load().oracle_nf4_storage_bytes(rows, cols, block, group, ctypes.byref(p),
                                          ctypes.byref(c), ctypes.byref(s))
    if rc != 0:
        raise ValueError("bad arguments")
    return p.value, c.value, s.value
