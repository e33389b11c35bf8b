"""Test-side helpers: error metrics, bf16 bit handling, nibble unpacking.

No arithmetic of the method lives here: quantisation, dequantisation and the
linear-layer contractions come from ``oracle/`` (expected values) or from the
CUDA library (values under test)."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances for floating-point outputs of the fused linear layer (bf16
# operands, fp32 accumulation) against the fp64 oracle.
MAX_ABS = 2e-2
REL_FRO = 1e-2


def to_np_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns (numpy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    """uint8 packed -> indices, element 2j from the high nibble of byte j."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.size * 2, dtype=np.uint8)
    out[0::2] = p >> 4
    out[1::2] = p & 0x0F
    return out


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    diff = got - ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(diff)) / den if den > 0 else float(np.linalg.norm(diff))
    return max_abs, rel


def assert_close(got, ref, what: str, max_abs: float = MAX_ABS, rel_fro: float = REL_FRO):
    ma, rf = errors(got, ref)
    assert ma <= max_abs and rf <= rel_fro, (
        f"{what}: max|err|={ma:.3e} (tol {max_abs:.0e}), rel-Frobenius={rf:.3e} (tol {rel_fro:.0e})")
    return ma, rf


def gemv_bound(x, w_hat) -> np.ndarray:
    """Per-output error bound of the decode GEMV against the exact-w_hat
    product: the GEMV scales each block's dot product of bf16 codepoints by
    the block constant instead of rounding every w_hat = bf16(c a_hat), so a
    term c' a_hat x differs from w_hat x by at most 2^-8 (1 + 2^-8) |w_hat x|
    (c' = bf16(c) and w_hat each within 2^-9 of c and c a_hat); the fp32
    accumulation (64 terms per block, then K/64 block sums) adds at most
    (K/64 + 66) 2^-23 of the same magnitude sum."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    w = np.abs(np.asarray(w_hat, dtype=np.float64))
    K = w.shape[1]
    return (2.0 ** -8 * (1 + 2.0 ** -8) + (K / 64 + 66) * 2.0 ** -23) * (x @ w.T)


def assert_close_bound(got, ref, bound, what: str, rel_fro: float = REL_FRO):
    """Every |got - ref| within its bound (plus 1e-5 |ref| + 1e-6 for the
    fp32 LoRA term), and the relative Frobenius error within rel_fro."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    lim = np.asarray(bound, dtype=np.float64) + 1e-5 * np.abs(ref) + 1e-6
    diff = np.abs(got - ref)
    bad = diff > lim
    ma, rf = errors(got, ref)
    assert not bad.any() and rf <= rel_fro, (
        f"{what}: {int(bad.sum())} outputs beyond their bound (worst |err|/bound "
        f"{float(np.max(diff / lim)):.3g}), rel-Frobenius={rf:.3e} (tol {rel_fro:.0e})")
    return ma, rf
