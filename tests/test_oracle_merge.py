"""Pins of the oracle's adapter merge, W_merged = bf16(W_hat + alpha/r B A)
("QLoRA and 4bit Quantization | QLoRA 与 4-bit 量化", Step 5 conclusion: the
merged adapter is what deployment loads).

  * the one rounding binary64 -> bf16 against brute force over exact
    rationals (ties to even, subnormal spacing);
  * B = 0 or A = 0 gives back the dequantised weight bit for bit;
  * the merged weight reproduces the forward pass: x W_merged^T (before
    rounding) equals the oracle's y = x W_hat^T + (x A^T) B^T alpha/r, which
    is itself pinned by torch fp64 autograd;
  * a hand example.
"""
from fractions import Fraction

import numpy as np

from oracle import oracle as orc


def _bf16_value(bits: int) -> Fraction:
    return Fraction(float(np.array([bits << 16], dtype=np.uint32).view(np.float32)[0]))


def _nearest_bf16_bruteforce(v: float) -> int:
    """Nearest bf16 to v by exact rationals; ties to the even pattern."""
    f = np.float32(v)
    c = int(np.array([f], dtype=np.float32).view(np.uint32)[0]) >> 16
    cands = {(c + d) & 0xFFFF for d in (-2, -1, 0, 1, 2)}
    cands = [b for b in cands if (b & 0x7F80) != 0x7F80]
    fv = Fraction(v)
    dist = {b: abs(_bf16_value(b) - fv) for b in cands}
    m = min(dist.values())
    best = [b for b, dd in dist.items() if dd == m]
    if len(best) > 1:
        best = [b for b in best if (b & 1) == 0]
    return best[0]


def test_double_to_bf16_rounding_matches_brute_force():
    rng = np.random.default_rng(3)
    vals = list(rng.standard_normal(400) * 0.05) + list(rng.standard_normal(100) * 1e-39)
    # exact ties between two bf16 values, both parities
    for b in (0x3F80, 0x3F81, 0xBC01, 0x3D00):
        lo, hi = _bf16_value(b), _bf16_value(b + 1)
        vals.append(float((lo + hi) / 2))
    vals += [0.0, 1.0, -2.5, 2.0 ** -130, -(2.0 ** -133) * 1.5]
    for v in vals:
        assert orc.bf16_rne_double(v) == _nearest_bf16_bruteforce(v), v


def _case(N=24, K=128, r=8, seed=0):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    q = orc.quantize_nf4(W, 64, 256)
    w_hat = orc.dequant_f32(q)
    A = orc.bf16_bits_to_f32(orc.bf16_rne(rng.standard_normal((r, K)) * 0.01)).reshape(r, K)
    B = orc.bf16_bits_to_f32(orc.bf16_rne(rng.standard_normal((N, r)) * 0.01)).reshape(N, r)
    return q, w_hat, A, B


def test_zero_factor_gives_the_dequantised_weight():
    q, w_hat, A, B = _case()
    deq = orc.dequant_bf16(q)
    for A_, B_ in ((A, np.zeros_like(B)), (np.zeros_like(A), B)):
        bits, exact = orc.merge_bf16(w_hat, A_, B_, 16.0)
        assert np.array_equal(bits, deq)
        assert np.array_equal(exact, w_hat.astype(np.float64))


def test_merged_weight_reproduces_the_forward():
    q, w_hat, A, B = _case(N=40, K=192, r=16, seed=1)
    alpha = 32.0
    x = orc.bf16_bits_to_f32(orc.bf16_rne(np.random.default_rng(2).standard_normal((5, 192))))
    x = x.reshape(5, 192)
    _, exact = orc.merge_bf16(w_hat, A, B, alpha)
    y_merged = x.astype(np.float64) @ exact.T
    y_ref, _ = orc.linear_fwd(x, w_hat, A, B, alpha)
    np.testing.assert_allclose(y_merged, y_ref, rtol=1e-12, atol=1e-12)


def test_hand_example():
    # 0.5 + (2/1) * 0.25 * 2 = 1.5; and a value that rounds: 0.1 + 2 * 0.5 * 0.001
    bits, exact = orc.merge_bf16(np.array([[0.5, 0.1]], np.float32),
                                 np.array([[2.0, 0.001]], np.float32),
                                 np.array([[0.25, ]], np.float32).reshape(1, 1), 2.0)
    assert exact[0, 0] == 1.5 and bits[0, 0] == 0x3FC0
    assert exact[0, 1] == float(np.float32(0.1)) + 2 * 0.25 * float(np.float32(0.001))
    assert bits[0, 1] == _nearest_bf16_bruteforce(exact[0, 1])
