"""Pins for the oracle's NF4 codebook and nearest-codepoint rule.

What pins them (nothing here re-derives the oracle's own code):
  * the 16 decimals printed on the pages (golden/nf4_codebook.txt);
  * the worked example 0.20 -> 0.161 (index 9) printed in the page text
    ("QLoRA and 4bit Quantization | QLoRA 与 4-bit 量化", Step 2);
  * the page's own codebook test (first entry negative, last positive, 16
    finite entries: Step 4, test_nf4_lookup_and_dequantization);
  * exact rational arithmetic (fractions.Fraction): the chosen codepoint must
    be a nearest codepoint of the value in exact arithmetic.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import oracle as orc


def _printed_table(golden_dir):
    vals = []
    with open(os.path.join(golden_dir, "nf4_codebook.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                vals.append(line)
    return vals


def test_codebook_equals_printed_decimals(golden_dir):
    printed = _printed_table(golden_dir)
    assert len(printed) == 16
    cb = orc.codebook()
    # binary32 nearest to each printed decimal (numpy parses with correct rounding)
    expect = np.array([np.float32(s) for s in printed], dtype=np.float32)
    assert cb.dtype == np.float32
    assert np.array_equal(cb.view(np.uint32), expect.view(np.uint32))


def test_codebook_invariants():
    cb = orc.codebook()
    assert cb.shape == (16,)
    assert np.all(np.isfinite(cb))
    assert np.all(np.diff(cb) > 0), "strictly increasing"
    assert cb[0] == -1.0 and cb[15] == 1.0 and cb[7] == 0.0
    assert cb[0] == -cb[15], "endpoint symmetry"
    assert cb[0] < 0 < cb[-1]
    # the printed table is NOT mirror-symmetric (7 negative, 8 positive); the
    # oracle must not "fix" that.
    assert (cb < 0).sum() == 7 and (cb > 0).sum() == 8
    assert cb[1] != -cb[14]


def test_codebook_is_not_the_quantile_formula():
    """Reading: the printed table is normative; the quantile formula of Step 2
    (q_i = inverse normal CDF of (i - 0.5)/16) gives a symmetric set with no
    exact zero, which does not reproduce the table."""
    from scipy.stats import norm
    q = norm.ppf((np.arange(1, 17) - 0.5) / 16)
    q = q / np.abs(q).max()
    cb = orc.codebook().astype(np.float64)
    assert not np.any(q == 0.0)
    assert np.max(np.abs(q - cb)) > 0.01


def test_worked_example(golden_dir):
    with open(os.path.join(golden_dir, "worked_example.json")) as f:
        ex = json.load(f)
    idx = orc.nearest_code(np.float32(ex["normalised_value"]))
    assert idx == ex["index_in_printed_table"]
    assert orc.codebook()[idx] == np.float32(ex["codepoint"])


def _exact_nearest_set(xn: np.float32, cb: np.ndarray):
    """All indices whose exact distance is within one binary32 rounding of
    the minimum (the fp32 distance rule may pick any of them)."""
    x = Fraction(float(xn))
    d = [abs(x - Fraction(float(c))) for c in cb]
    m = min(d)
    slack = Fraction(2) ** -24 * (m + abs(x) + 1)
    return {k for k, dk in enumerate(d) if dk - m <= slack}, d.index(m), m, d


def test_nearest_code_is_exact_nearest_on_random_values():
    rng = np.random.default_rng(123)
    cb = orc.codebook()
    xs = np.concatenate([
        rng.uniform(-1, 1, 4000).astype(np.float32),
        rng.normal(0, 0.3, 2000).clip(-1, 1).astype(np.float32),
    ])
    for xn in xs:
        got = orc.nearest_code(xn)
        ok, best, m, d = _exact_nearest_set(xn, cb)
        assert got in ok, (float(xn), got, best)
        if len(ok) == 1:
            assert got == best


def test_nearest_code_special_values():
    cb = orc.codebook()
    # every codepoint maps to itself
    for k, c in enumerate(cb):
        assert orc.nearest_code(c) == k
    # the ends of the normalised range
    assert orc.nearest_code(np.float32(1.0)) == 15
    assert orc.nearest_code(np.float32(-1.0)) == 0
    # zero and tiny values (denormals) map to the exact-zero codepoint
    for v in [0.0, -0.0, 1e-40, -1e-40, 1e-30, -1e-30]:
        assert orc.nearest_code(np.float32(v)) == 7
    # values next to each binary32 midpoint of neighbouring codepoints
    for k in range(15):
        mid = (np.float64(cb[k]) + np.float64(cb[k + 1])) / 2
        lo = np.nextafter(np.float32(mid), np.float32(-2))
        hi = np.nextafter(np.float32(mid), np.float32(2))
        for v in (lo, np.float32(mid), hi):
            got = orc.nearest_code(v)
            ok, best, _, _ = _exact_nearest_set(v, cb)
            assert got in ok and got in (k, k + 1)
        # clearly on either side
        assert orc.nearest_code(np.float32(mid - 1e-4)) == k
        assert orc.nearest_code(np.float32(mid + 1e-4)) == k + 1


def test_nearest_code_tie_goes_to_lower_index():
    """A binary32 value exactly halfway between two codepoints whose
    binary32 distances are equal must pick the lower index (reading)."""
    cb = orc.codebook()
    found = 0
    for k in range(15):
        a, b = np.float32(cb[k]), np.float32(cb[k + 1])
        mid = np.float32((np.float64(a) + np.float64(b)) / 2)
        for v in (np.nextafter(mid, np.float32(-2)), mid, np.nextafter(mid, np.float32(2))):
            # distances with binary32 subtraction (IEEE, as numpy performs it)
            da, db = abs(np.float32(v - a)), abs(np.float32(b - v))
            if da == db:
                found += 1
                assert orc.nearest_code(v) == k
    assert found >= 1, "expected at least one exact binary32 tie on the table"


def test_nearest_codes_bits_matches_scalar():
    start = np.float32(-0.3).view(np.uint32)
    out = orc.nearest_codes_bits(int(start), 1000)
    for i in range(0, 1000, 37):
        v = np.uint32(int(start) + i).view(np.float32)
        assert out[i] == orc.nearest_code(v)


def test_scaled_sweep_matches_block_quantisation():
    """The sweep helper (division by a block constant, then nearest code) gives
    the indices oracle_quantize_nf4 gives the same weights inside a block
    whose absmax is that constant; with absmax 1 it is the plain rule."""
    rng = np.random.default_rng(7)
    for a in (1.0, 0.0173, 3.3e-5, 2.0 ** -100, 1.7e3):
        a32 = np.float32(a)
        w = (rng.uniform(-1, 1, 63) * a32).astype(np.float32)
        start = int(np.float32(w[0]).view(np.uint32))
        block = np.concatenate([[a32], w]).astype(np.float32)
        q = orc.quantize_nf4(block.reshape(1, 64), 64, 0)
        for i in range(63):
            b = int(w[i].view(np.uint32))
            assert orc.nearest_codes_scaled_bits(b, 1, float(a32))[0] == q.idx[0, i + 1]
    bits = 0x3E000000
    assert np.array_equal(orc.nearest_codes_scaled_bits(bits, 4096, 1.0),
                          orc.nearest_codes_bits(bits, 4096))


# --------------------------------------------- quantile-formula codebook
# "QLoRA and 4bit Quantization | QLoRA 与 4-bit 量化", Step 2:
# q_i = Phi^-1((i - 0.5) / 16), i = 1..16, brought to [-1, 1] by q_16.

def test_inverse_normal_textbook_points():
    """Phi^-1 at points whose values are textbook: 0.5 -> 0, Phi(1) -> 1,
    Phi(2) -> 2, 0.975 -> 1.959963984540054; and scipy's ndtri (an
    independent implementation) at every p_i of the formula."""
    from scipy.special import ndtri
    assert abs(orc.inv_normal(0.5)) < 1e-12
    assert abs(orc.inv_normal(0.8413447460685429) - 1.0) < 1e-12
    assert abs(orc.inv_normal(0.9772498680518208) - 2.0) < 1e-12
    assert abs(orc.inv_normal(0.975) - 1.959963984540054) < 1e-12
    for i in range(1, 17):
        p = (i - 0.5) / 16
        assert abs(orc.inv_normal(p) - float(ndtri(p))) < 1e-12


def test_quantile_codebook_values_and_shape():
    """The table equals binary32(ndtri(p_i) / ndtri(p_16)) entry by entry, is
    exactly symmetric, strictly increasing, runs from -1 to 1 and has no zero
    (the nearest entries to zero are +-0.0421)."""
    from scipy.special import ndtri
    cb = orc.codebook(1)
    q16 = float(ndtri(15.5 / 16))
    expect = np.array([np.float32(float(ndtri((i - 0.5) / 16)) / q16) for i in range(1, 17)],
                      dtype=np.float32)
    assert np.array_equal(cb, expect)
    assert np.array_equal(cb, -cb[::-1])
    assert np.all(np.diff(cb) > 0) and cb[0] == -1.0 and cb[15] == 1.0
    assert not np.any(cb == 0.0)
    assert abs(cb[8] - 0.0421) < 5e-5


def test_quantile_codebook_quantisation_is_brute_force_nearest():
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((3, 128)) * 0.02).astype(np.float32)
    w[2, :64] = 0.0
    q = orc.quantize_nf4(w, 64, 0, codebook=1)
    cb = [Fraction(float(c)) for c in orc.codebook(1)]
    blocks, idx = w.reshape(-1, 64), q.idx.reshape(-1, 64)
    for b in range(blocks.shape[0]):
        a = Fraction(float(np.abs(blocks[b]).max()))
        for i in range(64):
            if a == 0:
                assert idx[b, i] == 7
                continue
            xn = Fraction(float(blocks[b, i])) / a
            d = [abs(xn - c) for c in cb]
            ok = {k for k, dk in enumerate(d) if dk - min(d) <= Fraction(2) ** -22}
            assert idx[b, i] in ok
    # the dequantised weight is the quantile codepoint times the constant
    deq = orc.dequant_f32(q)
    expect = orc.bf16_bits_to_f32(orc.bf16_rne(orc.codebook(1)[q.idx.ravel()] *
                                               np.repeat(q.absmax_f32, 64)))
    assert np.array_equal(deq.ravel(), expect)
