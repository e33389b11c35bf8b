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

